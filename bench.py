#!/usr/bin/env python3
"""Benchmark of the paged KV-cache attention path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload all|mha|gqa|long|mixed|tiny|swap]

One step = one pass of the whole hot path over one batch: the new token's
K/V of every sequence is written through its slot (slots from
pa_slot_mapping over the batch's block table), then single-query paged
attention runs over every sequence (and the partition merge where a sequence
was split); for the mixed batch, every new token's K/V is written, then
pa_varlen_mixed attends all query rows (its prefill sequences through the
varlen tensor-core kernel, its trailing one-token sequences through the
decode kernel; the one-call pa_prefill_varlen form is reported beside).

The default (--workload all) prints ONE JSON line: the headline workload, the
7B-shaped MHA decode layer (64 sequences, 32 heads, head size 128, block size
16, fp16, attended lengths uniform in [1, 2048], physical blocks drawn from a
seeded permutation of a 10,000-block pool), and under "configs" one record
per other workload -- the worked example ("tiny"), the GQA parallel-sampling
batch built through the library's block pool, fork and copy-on-write ("gqa"),
the long-context E4M3 split-K decode ("long") and the mixed varlen prefill +
decode batch ("mixed") -- each with its own value, roofline, e2e, clocks and
CPU baseline.  The GQA batch's attention call is pa_decode_cascade (its
groups share their prompt blocks); the plain pa_decode step is reported
beside it.

`value` is the algorithmic K/V bytes the step reads (sum over sequences of
L * num_kv_heads * head_size * 2 * element size) per second of device time,
summed over ranks, with all inputs resident in HBM (the mixed batch: causal
FLOPs per second).  `e2e` is the same metric when every step also copies its
inputs from pinned host memory and reads the outputs back.  With N > 1
(torchrun) every rank runs its own replica: the path has no exchange step, so
there is no collective in the timed work.

--impl reference times the CPU oracle (test infrastructure) on the host cores
on a bounded sample of the same workload.
"""
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
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_75_gb300 import workloads as W  # noqa: E402

METRIC = "paged-attn decode KV-read GB/s (% of GB300 HBM peak); decode seqs/s per layer"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

# DRAM bytes (read + write) per launch of the dominant kernel, from one ncu
# capture per workload, listed in profiles/ncu_traffic.md as table rows
# "| workload | kernel source hash | bytes | ..."; a figure is reported only
# while the kernel source it was taken on is unchanged.
TRAFFIC_TABLE = os.path.join(ROOT, "profiles", "ncu_traffic.md")


def ncu_traffic(workload, src_hash):
    try:
        with open(TRAFFIC_TABLE) as f:
            for line in f:
                cells = [c.strip() for c in line.strip().strip("|").split("|")]
                if len(cells) >= 3 and cells[0] == workload and cells[1] == src_hash:
                    return int(cells[2].replace(",", "").replace("_", ""))
    except OSError:
        pass
    return None


L2_BYTES = 129 * 1024 * 1024
# nominal host link of a Grace-Blackwell superchip (NVLink-C2C), per direction
C2C_GBS_PER_DIRECTION = 450.0
DECODE_SOURCES = ("decode_impl.cuh", "decode_launch.cuh", "decode_api.cu", "common.cuh")
PREFILL_SOURCES = ("prefill.cu", "common.cuh", "launch.h")


def kernel_source_hash(files=DECODE_SOURCES):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "paged_kv_cache_75_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


class L2Flush:
    """Writes a buffer twice the size of L2 between timed iterations when the
    inputs alone would fit in L2; the flush itself is outside every timed
    interval."""

    def __init__(self, device, needed):
        self.buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=device) if needed else None

    def __call__(self):
        if self.buf is not None:
            self.buf.fill_(1)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region (NVML through ctypes; nvidia-smi fallback)
# ---------------------------------------------------------------------------
REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
           0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
           0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}


class ClockSampler:
    def __init__(self, device_index=0, period_s=0.01):
        self.samples, self.reasons, self.max_mhz = [], 0, None
        self.period = period_s
        self._stop = threading.Event()
        self._nvml = None
        self._handle = ctypes.c_void_p()
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit")
            props = torch.cuda.get_device_properties(device_index)
            bus = "%08x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id, props.pci_device_id)
            if nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self._handle)) != 0:
                if nv.nvmlDeviceGetHandleByIndex_v2(device_index, ctypes.byref(self._handle)) != 0:
                    raise OSError("nvml handle")
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(self._handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._nvml = nv
        except Exception:
            self._nvml = None
        self._thread = threading.Thread(target=self._run, daemon=True)

    def _sample(self):
        if self._nvml is not None:
            mhz, rs = ctypes.c_uint(), ctypes.c_ulonglong()
            self._nvml.nvmlDeviceGetClockInfo(self._handle, 1, ctypes.byref(mhz))
            f = getattr(self._nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                self._nvml.nvmlDeviceGetCurrentClocksThrottleReasons
            f(self._handle, ctypes.byref(rs))
            return mhz.value, rs.value
        out = subprocess.run(["nvidia-smi", "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                              "--format=csv,noheader,nounits", "-i", "0"], capture_output=True, text=True,
                             timeout=5).stdout.strip().split(",")
        if self.max_mhz is None:
            self.max_mhz = int(out[1])
        return int(out[0]), int(out[2].strip(), 16)

    def _run(self):
        while not self._stop.is_set():
            try:
                mhz, rs = self._sample()
                self.samples.append(mhz)
                self.reasons |= rs
            except Exception:
                pass
            self._stop.wait(self.period)

    def __enter__(self):
        self._thread.start()
        return self

    def __exit__(self, *exc):
        try:
            mhz, rs = self._sample()  # at least one sample at the end of the region
            self.samples.append(mhz)
            self.reasons |= rs
        except Exception:
            pass
        self._stop.set()
        self._thread.join()

    def summary(self):
        names = [n for b, n in REASONS.items() if self.reasons & b and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": names, "samples": len(self.samples)}


# ---------------------------------------------------------------------------
# multi-process helpers (replicas; no collective in the timed work)
# ---------------------------------------------------------------------------
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def aggregate(elapsed_ms: float, units: float, world: int):
    """(max elapsed over ranks, sum of units over ranks)."""
    if world == 1:
        return elapsed_ms, units
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
class DecodeStep:
    """Inputs of one decode step resident on the device."""

    def __init__(self, case: W.PagedCase, device, partition_size=0, name=""):
        import paged_kv_cache_75_gb300 as pk
        self.pk = pk
        self.name = name
        self.case = case
        self.device = device
        lens = case.seq_lens.cpu().numpy().astype(np.int64)
        self.lens_np = lens
        B = len(lens)
        self.B = B
        # a1: the slot of each sequence's newest token (position L-1)
        bt = case.block_table.cpu().numpy()
        self.slots_np = pk.pa_slot_mapping(bt, case.block_size, np.arange(B, dtype=np.int32), lens - 1)
        g = torch.Generator(device=device)
        g.manual_seed(12345)
        self.k_new = W.random_values(g, (B, case.num_kv_heads, case.head_size), case.q_dtype, device)
        self.v_new = W.random_values(g, (B, case.num_kv_heads, case.head_size), case.q_dtype, device)
        self.slots = torch.from_numpy(self.slots_np).to(device)
        self.cache = pk.KVCache(case.k_cache, case.v_cache, case.k_scale, case.v_scale)
        self.q = case.q
        self.bt = case.block_table.to(device)
        self.lens = case.seq_lens.to(device)
        self.max_len = int(lens.max())
        self.P = partition_size
        self.out = torch.empty_like(self.q)
        ws = pk.pa_decode_workspace_size(B, case.num_heads, case.head_size, self.max_len, case.block_size,
                                         partition_size)
        self.ws = torch.empty(max(ws, 16), dtype=torch.uint8, device=device)
        self.kv_bytes = case.kv_bytes()
        P = partition_size or pk.pa_decode_partition_size(B, case.num_heads, case.num_kv_heads, self.max_len)
        self.P_eff = P
        self.split = self.max_len > P
        self.launches_per_step = 2 + (1 if self.split else 0)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.has_groups = "cu_groups" in case.meta
        if self.has_groups:
            self.launches_per_step = 3  # write, the group-mode decode, the merge
        if self.has_groups:
            cu, sl = case.meta["cu_groups"], case.meta["shared_lens"]
            self.cu_groups = torch.as_tensor(cu).to(device)
            self.shared_lens = torch.as_tensor(sl).to(device)
            self.max_group = int(np.diff(cu).max())
            self.max_shared = int(sl.max())
            nws = pk.pa_decode_cascade_workspace_size(B, case.num_heads, case.head_size, self.max_len,
                                                      case.block_size, partition_size)
            self.ws_cascade = torch.empty(nws, dtype=torch.uint8, device=device)

    def write(self):
        self.pk.pa_kv_cache_write(self.cache, self.k_new, self.v_new, self.slots, self.status)

    def append(self):
        """The same step through pa_decode_append: write and attend in one launch."""
        self.pk.pa_decode_append(self.out, self.q, self.k_new, self.v_new, self.cache, self.bt, self.lens,
                                 self.max_len, self.case.scale, self.P, self.ws, self.status)

    def cascade(self):
        """The same step's attention through pa_decode_cascade (the workload's
        sampling groups read their shared prompt blocks once)."""
        self.pk.pa_decode_cascade(self.out, self.q, self.cache, self.bt, self.lens, self.max_len, self.case.scale,
                                  self.cu_groups, self.shared_lens, self.max_group, self.max_shared, self.ws_cascade,
                                  self.P, self.status)

    def decode(self, q=None, out=None, bt=None, lens=None):
        self.pk.pa_decode(self.out if out is None else out, self.q if q is None else q, self.cache,
                          self.bt if bt is None else bt, self.lens if lens is None else lens, self.max_len,
                          self.case.scale, self.P, self.ws, self.status)

    def attend(self, q=None, out=None, bt=None, lens=None, cu_groups=None, shared_lens=None):
        """The step's attention call: pa_decode_cascade for a batch of sampling
        groups that share their prompt blocks (the library's call for such a
        batch), pa_decode otherwise."""
        if not self.has_groups:
            return self.decode(q, out, bt, lens)
        self.pk.pa_decode_cascade(self.out if out is None else out, self.q if q is None else q, self.cache,
                                  self.bt if bt is None else bt, self.lens if lens is None else lens, self.max_len,
                                  self.case.scale, self.cu_groups if cu_groups is None else cu_groups,
                                  self.shared_lens if shared_lens is None else shared_lens, self.max_group,
                                  self.max_shared, self.ws_cascade, self.P, self.status)


class PrefillStep:
    """Inputs of one mixed varlen step (new tokens' K/V written through their
    slots, then attention over all sequences: through pa_varlen_mixed, which
    sends the prefill sequences to the varlen kernel and the trailing
    one-token sequences to the decode kernel, or as one pa_prefill_varlen
    call over all of them), on the device."""

    def __init__(self, case: W.PagedCase, device, name=""):
        import paged_kv_cache_75_gb300 as pk
        self.pk = pk
        self.name = name
        self.case = case
        self.device = device
        lq = np.asarray(case.meta["query_lens"], np.int64)
        lk = np.asarray(case.meta["key_lens"], np.int64)
        self.lq, self.lk = lq, lk
        self.B = len(lq)
        bt = case.block_table.cpu().numpy()
        # a1: slots of each sequence's new tokens, positions Lk-Lq .. Lk-1
        seq_idx = np.repeat(np.arange(self.B, dtype=np.int32), lq)
        pos = np.concatenate([np.arange(k - q, k) for q, k in zip(lq, lk)]).astype(np.int64)
        self.slots = torch.from_numpy(pk.pa_slot_mapping(bt, case.block_size, seq_idx, pos)).to(device)
        T = int(lq.sum())
        g = torch.Generator(device=device)
        g.manual_seed(54321)
        self.k_new = W.random_values(g, (T, case.num_kv_heads, case.head_size), case.q_dtype, device)
        self.v_new = W.random_values(g, (T, case.num_kv_heads, case.head_size), case.q_dtype, device)
        self.cache = pk.KVCache(case.k_cache, case.v_cache)
        self.q = case.q
        self.bt = case.block_table.to(device)
        self.cu_q = case.cu_seq_lens_q.to(device)
        self.cu_k = case.cu_seq_lens_k.to(device)
        self.max_q, self.max_k = int(lq.max()), int(lk.max())
        self.out = torch.empty_like(self.q)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        # algorithmic FLOPs: 4 * D * H per visible (query, key) pair, causal
        pairs = 0
        for q, k in zip(lq, lk):
            i = np.arange(q)
            pairs += int(np.minimum(k, k - q + i + 1).clip(min=0).sum())
        self.flops = 4 * case.head_size * case.num_heads * pairs
        self.pairs = pairs
        # the mixed dispatcher: the trailing run of one-token sequences goes
        # to the decode kernel, the rest to the varlen kernel
        self.host_cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
        n_dec = 0
        while n_dec < self.B and lq[self.B - 1 - n_dec] == 1:
            n_dec += 1
        self.n_pre = self.B - n_dec
        pre_pairs = 0
        for q, k in zip(lq[:self.n_pre], lk[:self.n_pre]):
            i = np.arange(q)
            pre_pairs += int(np.minimum(k, k - q + i + 1).clip(min=0).sum())
        self.prefill_flops = 4 * case.head_size * case.num_heads * pre_pairs
        self.max_q_pre = int(lq[:self.n_pre].max()) if self.n_pre else 0
        self.max_k_pre = int(lk[:self.n_pre].max()) if self.n_pre else 0
        ws_n = pk.pa_varlen_mixed_workspace_size(self.B, case.num_heads, case.head_size, self.max_k,
                                                 case.block_size)
        self.ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=device)
        dec_P = pk.pa_decode_partition_size(max(n_dec, 1), case.num_heads, case.num_kv_heads, self.max_k)
        # write, the varlen kernel, the decode kernel (and its merge when a
        # one-token sequence spans several partitions)
        self.launches_per_step = 1 + (1 if self.n_pre else 0) + (
            (2 if self.max_k > dec_P else 1) if n_dec else 0)

    def write(self):
        self.pk.pa_kv_cache_write(self.cache, self.k_new, self.v_new, self.slots, self.status)

    def mixed(self, q=None, out=None, cu_q=None, cu_k=None, bt=None):
        """The step's attention: pa_varlen_mixed."""
        self.pk.pa_varlen_mixed(self.out if out is None else out, self.q if q is None else q, self.cache,
                                self.bt if bt is None else bt, self.cu_q if cu_q is None else cu_q,
                                self.cu_k if cu_k is None else cu_k, self.host_cu_q, self.max_q, self.max_k,
                                self.case.scale, True, self.ws, self.status)

    def main(self, q=None, out=None):
        """One pa_prefill_varlen call over every sequence."""
        self.pk.pa_prefill_varlen(self.out if out is None else out, self.q if q is None else q, self.cache,
                                  self.bt, self.cu_q, self.cu_k, self.max_q, self.max_k, self.case.scale, True,
                                  self.status)

    def prefill_rows(self):
        """The varlen kernel alone on the prefill sequences (the launch
        pa_varlen_mixed makes for them)."""
        n = self.n_pre
        self.pk.pa_prefill_varlen(self.out, self.q, self.cache, self.bt[:n], self.cu_q[:n + 1], self.cu_k[:n + 1],
                                  self.max_q_pre, self.max_k_pre, self.case.scale, True, self.status)


def build_workload(name, device, num_seqs=None, pool_blocks=None):
    if name == "mha":
        B = num_seqs or 64
        nb = pool_blocks or 10_000
        tag = "mha_decode_%dseq_32h_d128_bs16_fp16_len_u1_2048_pool%d" % (B, nb)
        return W.mha_decode(device=device, B=B, num_blocks=nb), tag
    if name == "gqa":
        from paged_kv_cache_75_gb300 import sampling
        groups = (num_seqs or 256) // 4
        case = sampling.build_sampled_batch(W.gqa_sampling_inputs(device=device, groups=groups), device)
        torch.cuda.synchronize()
        if int(case.meta["dev_status"].item()) != 0:
            raise RuntimeError("device status %d while building the sampled batch"
                               % int(case.meta["dev_status"].item()))
        return case, build_workload_name("gqa", groups)
    if name == "long":
        B = num_seqs or 8
        return W.long_fp8_decode(device=device, B=B), "long_decode_%dseq_64q8kv_d128_bs32_e4m3_len_u32k_128k_p512" % B
    if name == "mixed":
        return W.mixed_varlen(device=device), "mixed_varlen_8prefill_120decode_32q8kv_d128_bs16_bf16_causal"
    if name == "tiny":
        case = W.tiny_decode(device=device)
        case.seq_lens = torch.tensor([31, 33, 71], dtype=torch.int32, device=device)
        return case, "tiny_decode_3seq_4h_d64_bs32_fp16_worked_example"
    raise ValueError(name)


def unique_bytes_of(case):
    return case.unique_kv_bytes()


def kernel_pass(stream, steps, before, kernel, flush=None):
    """Mean ms of `kernel` over `steps` launches, each bracketed by CUDA events
    on `stream` with `before` (the step's other launches) ahead of it.  An
    event between two launches ends their programmatic overlap, so this pass
    runs after the timed steps, not inside them."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        if flush is not None:
            flush()
        before()
        evs[i][0].record(stream)
        kernel()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / steps


def timed_decode(step: DecodeStep, steps, warmup, world, flush, attend=None):
    """Returns (total ms over the timed steps, mean decode-kernel ms, clocks).
    The timed steps (write + decode) carry no event between their launches;
    with an L2 flush every step is timed on its own and the flush runs between
    the timed intervals.  The decode kernel's own duration comes from a second
    pass over the same steps with events around each decode launch; clocks are
    sampled over both."""
    stream = torch.cuda.current_stream()
    attend = step.attend if attend is None else attend
    for _ in range(warmup):
        step.write()
        attend()
    torch.cuda.synchronize()
    whole = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        start.record(stream)
        for i in range(steps):
            if flush.buf is not None:
                flush()
                whole[i][0].record(stream)
            step.write()
            attend()
            if flush.buf is not None:
                whole[i][1].record(stream)
        end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        decode_ms = kernel_pass(stream, steps, step.write, attend, flush if flush.buf is not None else None)
    total_ms = sum(a.elapsed_time(b) for a, b in whole) if flush.buf is not None else start.elapsed_time(end)
    st = int(step.status.item())
    if st != 0:
        raise RuntimeError("device status %d during the benchmark" % st)
    return total_ms, decode_ms, clk.summary()


def timed_append(step: DecodeStep, steps, warmup, flush):
    """Mean ms of one fused step (pa_decode_append), each step timed on its
    own with the L2 flush (if any) outside the timed interval."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        step.append()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush()
        evs[i][0].record(stream)
        step.append()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    if int(step.status.item()) != 0:
        raise RuntimeError("device status %d in the fused step" % int(step.status.item()))
    return sum(a.elapsed_time(b) for a, b in evs) / steps


def timed_graph(step: DecodeStep, steps, flush):
    """One step (write + decode) captured as a CUDA graph and replayed: the
    device-side latency without host launch overhead.  Each replay is timed on
    its own, the L2 flush runs between replays."""
    stream = torch.cuda.current_stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step.write()
        step.attend()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush()
        evs[i][0].record(stream)
        graph.replay()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / steps


def timed_prefill(step: PrefillStep, steps, warmup, world, attend, kernel):
    """Returns (total ms over the timed steps, mean varlen-kernel ms, clocks):
    the timed steps (write + `attend`) carry no event between their launches;
    the varlen kernel's own duration comes from a second pass with events
    around each `kernel` call."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        step.write()
        attend()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        start.record(stream)
        for i in range(steps):
            step.write()
            attend()
        end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        kernel_ms = kernel_pass(stream, steps, step.write, kernel)
    st = int(step.status.item())
    if st != 0:
        raise RuntimeError("device status %d during the benchmark" % st)
    return start.elapsed_time(end), kernel_ms, clk.summary()


E2E_NOTE = ("double-buffered: step i+1's inputs go up on one copy stream while step i computes, "
            "step i's output comes back on another; the host waits for each step's output one step later; "
            "every step's copies are inside the timed region")


def pipelined_e2e(device, src, out_like, launch, steps, warmup, world):
    """End-to-end steps through the public API with host buffers, as a serving
    loop runs them: every step copies its inputs (`src`, packed into one
    page-locked buffer of 16-byte-aligned pieces) to the device and its output
    back to page-locked host memory.  Two device copies of the inputs and of
    the output let step i+1's upload and step i-1's download overlap step i's
    kernels; the host waits for each step's output one step later.
    `launch(views, out)` issues a step's library calls on the current stream.
    Returns (ms for `steps` steps, H2D bytes per step, D2H bytes per step)."""
    offs, total = {}, 0
    for n, t in src:
        offs[n] = total
        total += (t.numel() * t.element_size() + 15) // 16 * 16
    host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()

    def view(buf, n, t):
        nbytes = t.numel() * t.element_size()
        return buf[offs[n]:offs[n] + nbytes].view(t.dtype).view(t.shape)

    for n, t in src:
        view(host_buf, n, t).copy_(t.cpu())
    dev_bufs = [torch.empty(total, dtype=torch.uint8, device=device) for _ in range(2)]
    views = [{n: view(buf, n, t) for n, t in src} for buf in dev_bufs]
    outs = [torch.empty_like(out_like) for _ in range(2)]
    out_host = [torch.empty(out_like.shape, dtype=out_like.dtype).pin_memory() for _ in range(2)]
    comp = torch.cuda.current_stream(device)
    up, down = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def upload(i):
        b = i % 2
        up.wait_event(ev_done[b])  # step i-2 has finished with these inputs
        with torch.cuda.stream(up):
            dev_bufs[b].copy_(host_buf, non_blocking=True)
        ev_in[b].record(up)

    def run(n, start=None):
        if start is not None:
            up.wait_event(start)
        upload(0)
        for i in range(n):
            b = i % 2
            comp.wait_event(ev_in[b])
            comp.wait_event(ev_out[b])  # step i-2's output has been read back
            launch(views[b], outs[b])
            ev_done[b].record(comp)
            if i + 1 < n:
                upload(i + 1)
            down.wait_event(ev_done[b])
            with torch.cuda.stream(down):
                out_host[b].copy_(outs[b], non_blocking=True)
            ev_out[b].record(down)
            if i >= 1:
                ev_out[(i - 1) % 2].synchronize()  # the host takes step i-1's output
        comp.wait_event(ev_out[(n - 1) % 2])

    run(warmup)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(comp)
    run(steps, start)
    end.record(comp)
    end.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    h2d = total
    d2h = out_like.numel() * out_like.element_size()
    return start.elapsed_time(end), h2d, d2h


def timed_prefill_e2e(step: PrefillStep, steps, warmup, world):
    """The mixed step end to end: q, the new K/V, slots, cumulative lengths and
    block table up from page-locked host memory, the output back."""
    src = (("q", step.q), ("k", step.k_new), ("v", step.v_new), ("slots", step.slots), ("cu_q", step.cu_q),
           ("cu_k", step.cu_k), ("bt", step.bt))
    pk = step.pk

    def launch(dev, out):
        pk.pa_kv_cache_write(step.cache, dev["k"], dev["v"], dev["slots"], step.status)
        step.mixed(q=dev["q"], out=out, cu_q=dev["cu_q"], cu_k=dev["cu_k"], bt=dev["bt"])

    return pipelined_e2e(step.device, src, step.out, launch, steps, warmup, world)


def run_prefill(args, case, wname, dev, rank, world, cpu_budget=10.0):
    step = PrefillStep(case, dev, wname)
    # the step: new K/V written, then pa_varlen_mixed; the dominant kernel is
    # the varlen kernel on the prefill sequences
    total_ms, main_ms, clocks = timed_prefill(step, args.steps, args.warmup, world, step.mixed, step.prefill_rows)
    total_ms, flops_sum = aggregate(total_ms, float(step.flops) * args.steps, world)
    e2e_ms, h2d, d2h = timed_prefill_e2e(step, args.steps, args.warmup, world)
    e2e_ms, flops_e2e = aggregate(e2e_ms, float(step.flops) * args.steps, world)
    # the same step as one pa_prefill_varlen call over all 128 sequences
    one_ms, one_kernel_ms, _ = timed_prefill(step, args.steps, args.warmup, world, step.main, step.main)
    one_ms, one_sum = aggregate(one_ms, float(step.flops) * args.steps, world)
    _, tflops_peak, tflops_sustained, peak_kind = measured_peaks()
    # the varlen kernel is timed per launch in steps of well under a
    # millisecond, not inside a seconds-long loop: the burst peak applies
    achieved = step.prefill_flops / (main_ms / 1e3) / 1e12
    one_achieved = step.flops / (one_kernel_ms / 1e3) / 1e12
    line = {
        "metric": "paged-attn varlen prefill TFLOP/s (causal, % of GB300 bf16 tensor peak)",
        "value": round(flops_sum / (total_ms / 1e3) / 1e12, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {0: "f16", 1: "bf16"}[case.q_dtype],
        "accumulate": "f32",
        "data": "synthetic",
        "config": {"workload": wname, "num_seqs": step.B, "num_heads": case.num_heads,
                   "num_kv_heads": case.num_kv_heads, "head_size": case.head_size, "block_size": case.block_size,
                   "total_q": int(step.lq.sum()), "visible_pairs": step.pairs, "flops_per_step": step.flops,
                   "prefill_seqs": step.n_pre, "prefill_flops_per_step": step.prefill_flops,
                   "l2": "inputs larger than L2 (%.2f GB of K/V cache)" % (
                       2 * case.k_cache.numel() * case.k_cache.element_size() / 1e9),
                   "parallelism": "replicas" if world > 1 else "single"},
        "attention_call": "pa_varlen_mixed",
        "clocks": clocks,
        "e2e": {"value": round(flops_e2e / (e2e_ms / 1e3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms / args.steps, 5), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "pipeline": E2E_NOTE},
        "gpu_launches": step.launches_per_step * args.steps,
        "one_varlen_call": {
            "ms_per_step": round(one_ms / args.steps, 5), "value": round(one_sum / (one_ms / 1e3) / 1e12, 2),
            "unit": "TFLOP/s", "kernel_achieved": round(one_achieved, 2),
            "kernel_frac": round(one_achieved / tflops_peak, 4),
            "note": "the same step with the attention as one pa_prefill_varlen call over all 128 sequences (the "
                    "one-token rows as 128-row tiles with four live rows); not in value"},
        "roofline": {"bound": "tensor",
                     "kernel": "paged_prefill_tc_kernel (pa_varlen_mixed's launch over the 8 prefill sequences)",
                     "achieved": round(achieved, 2), "peak": tflops_peak, "unit": "TFLOP/s",
                     "frac": round(achieved / tflops_peak, 4),
                     "flops": "causal FLOPs of the prefill sequences (prefill_flops_per_step)",
                     "peak_kind": "of %s (bf16 dense, burst)" % peak_kind,
                     "frac_of_sustained": round(achieved / tflops_sustained, 4),
                     "traffic": ncu_traffic("mixed_prefill_rows", kernel_source_hash(PREFILL_SOURCES)),
                     "prefill_ms": round(main_ms, 5), "kernel_src": kernel_source_hash(PREFILL_SOURCES)},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_prefill(case, cpu_budget)
    return line


def timed_e2e(step: DecodeStep, steps, warmup, world):
    """The decode step end to end: q, the new K/V, slots, block table and
    lengths up from page-locked host memory, the output back."""
    src = [("q", step.q), ("k", step.k_new), ("v", step.v_new), ("slots", step.slots), ("bt", step.bt),
           ("lens", step.lens)]
    if step.has_groups:
        src += [("cu_groups", step.cu_groups), ("shared_lens", step.shared_lens)]
    pk = step.pk

    def launch(dev, out):
        pk.pa_kv_cache_write(step.cache, dev["k"], dev["v"], dev["slots"], step.status)
        step.attend(q=dev["q"], out=out, bt=dev["bt"], lens=dev["lens"], cu_groups=dev.get("cu_groups"),
                    shared_lens=dev.get("shared_lens"))

    return pipelined_e2e(step.device, src, step.out, launch, steps, warmup, world)


def oracle_decode_seconds(case: W.PagedCase, seq_idx, nthreads, q_bits, kc, vc, bt, lens):
    import oracle
    idx = np.asarray(seq_idx)
    t0 = time.perf_counter()
    _, _, rc = oracle.decode(q_bits[idx], case.q_dtype, kc, vc, case.kv_dtype, bt[idx], lens[idx], case.scale,
                             case.k_scale, case.v_scale, nthreads=nthreads, want_codes=True)
    dt = time.perf_counter() - t0
    assert rc == 0
    return dt


def cpu_sample_indices(case, budget_bytes):
    """Every k-th sequence so that the sample's KV bytes stay within budget."""
    lens = case.seq_lens.cpu().numpy().astype(np.int64)
    per = case.num_kv_heads * case.head_size * 2 * W.ELEM_BYTES[case.kv_dtype]
    total = int(lens.sum()) * per
    k = max(1, int(np.ceil(total / budget_bytes)))
    idx = np.arange(0, len(lens), k)
    return idx, int(lens[idx].sum()) * per


def cpu_baseline(case, budget_s=10.0):
    """The oracle, as it stands, on all host cores over a bounded sample."""
    import oracle
    cores = os.cpu_count() or 1
    n = oracle.num_threads(cores)
    q_bits, kc, vc = W.as_bits(case.q), W.as_bits(case.k_cache), W.as_bits(case.v_cache)
    bt = case.block_table.cpu().numpy()
    lens = case.seq_lens.cpu().numpy()
    idx, sample_bytes = cpu_sample_indices(case, 2e9)
    reps, spent = 0, 0.0
    while spent < budget_s and reps < 50:
        spent += oracle_decode_seconds(case, idx, n, q_bits, kc, vc, bt, lens)
        reps += 1
    gbs = sample_bytes * reps / spent / 1e9
    return {"value": round(gbs, 3), "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": "oracle decode (fp64) over %d of %d sequences (%.1f MB of KV), %d passes in %.1f s"
                      % (len(idx), case.num_seqs, sample_bytes / 1e6, reps, spent)}


def prefill_sample(case, rows_per_prefill=16, decode_every=6):
    """A valid sub-batch of a varlen case: the last rows of every prefill
    sequence (bottom-right alignment keeps them exact) and every k-th decode
    sequence.  Returns (q codes, table, cu_q, cu_k, visible pairs)."""
    lq = np.asarray(case.meta["query_lens"], np.int64)
    lk = np.asarray(case.meta["key_lens"], np.int64)
    n_pre = int(case.meta["n_prefill"])
    cu_q = case.cu_seq_lens_q.cpu().numpy()
    q_bits = W.as_bits(case.q)
    bt = case.block_table.cpu().numpy()
    seqs = list(range(n_pre)) + list(range(n_pre, len(lq), decode_every))
    rows, sq, sk, tab = [], [0], [0], []
    pairs = 0
    for b in seqs:
        r = int(min(lq[b], rows_per_prefill))
        rows.extend(range(int(cu_q[b + 1]) - r, int(cu_q[b + 1])))
        sq.append(sq[-1] + r)
        sk.append(sk[-1] + int(lk[b]))
        tab.append(bt[b])
        i = np.arange(lq[b] - r, lq[b])
        pairs += int(np.minimum(lk[b], lk[b] - lq[b] + i + 1).clip(min=0).sum())
    return (q_bits[np.asarray(rows)], np.stack(tab), np.asarray(sq, np.int32), np.asarray(sk, np.int32), pairs)


def oracle_prefill_seconds(case, sample, nthreads, kc, vc):
    import oracle
    qs, tab, sq, sk, _ = sample
    t0 = time.perf_counter()
    _, _, rc = oracle.prefill(qs, case.q_dtype, kc, vc, case.kv_dtype, tab, sq, sk, case.scale, True,
                              nthreads=nthreads)
    dt = time.perf_counter() - t0
    assert rc == 0
    return dt


def cpu_baseline_prefill(case, budget_s=10.0):
    """The oracle's varlen prefill, as it stands, on all host cores over a
    bounded sub-batch of the same workload, in the metric's unit."""
    import oracle
    n = oracle.num_threads(os.cpu_count() or 1)
    kc, vc = W.as_bits(case.k_cache), W.as_bits(case.v_cache)
    sample = prefill_sample(case)
    flops = 4 * case.head_size * case.num_heads * sample[4]
    reps, spent = 0, 0.0
    while spent < budget_s and reps < 50:
        spent += oracle_prefill_seconds(case, sample, n, kc, vc)
        reps += 1
    return {"value": round(flops * reps / spent / 1e12, 6), "unit": "TFLOP/s", "cores": n, "kind": "oracle",
            "sample": "oracle varlen prefill (fp64) over the last 16 query rows of each prefill sequence and "
                      "every 6th decode sequence (%d rows, %.2f GFLOP), %d passes in %.1f s"
                      % (int(sample[2][-1]), flops / 1e9, reps, spent)}


def run_swap(args, dev, rank, world):
    """Swap-based preemption's data move: whole blocks of an MHA-shaped cache
    (32 KV heads x 16 tokens x 128 fp16, K and V: 256 KiB a block) out to
    page-locked host memory and back in one pa_swap_blocks call each way.
    Roofline: a single contiguous copy of the same bytes between the same
    memories (cudaMemcpyAsync through torch), measured in the same run."""
    import paged_kv_cache_75_gb300 as pk
    nb, hkv, bs, d, n = 10_000, 32, 16, 128, 4096
    g = torch.Generator(device=dev)
    g.manual_seed(777)
    k = torch.empty((nb, hkv, bs, d), dtype=torch.float16, device=dev).normal_(generator=g)
    v = torch.empty_like(k).normal_(generator=g)
    cache = pk.KVCache(k, v)
    hk = torch.empty((n, hkv, bs, d), dtype=torch.float16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    rng = np.random.default_rng(778)
    dev_ids = rng.permutation(nb)[:n].astype(np.int32)
    pairs = torch.from_numpy(np.stack([dev_ids, np.arange(n, dtype=np.int32)], 1).copy()).to(dev)
    back = torch.from_numpy(np.stack([rng.permutation(nb)[:n].astype(np.int32),
                                      np.arange(n, dtype=np.int32)], 1).copy()).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    bytes_one_way = 2 * n * hkv * bs * d * 2
    stream = torch.cuda.current_stream()

    def timed(fn, steps):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i in range(steps):
            evs[i][0].record(stream)
            fn()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in evs) / steps

    out = lambda: pk.pa_swap_blocks(cache, hk, hv, pairs, True, status)
    inn = lambda: pk.pa_swap_blocks(cache, hk, hv, back, False, status)
    flat_d = torch.empty(bytes_one_way, dtype=torch.uint8, device=dev)
    flat_h = torch.empty(bytes_one_way, dtype=torch.uint8).pin_memory()
    d2h = lambda: flat_h.copy_(flat_d, non_blocking=True)
    h2d = lambda: flat_d.copy_(flat_h, non_blocking=True)
    for f in (out, inn, d2h, h2d):
        for _ in range(args.warmup):
            f()
    torch.cuda.synchronize()
    steps = max(3, min(args.steps, 50))
    barrier(world)
    with ClockSampler(torch.cuda.current_device()) as clk:
        t_out, t_in = timed(out, steps), timed(inn, steps)
    t_d2h, t_h2d = timed(d2h, steps), timed(h2d, steps)
    barrier(world)
    if int(status.item()) != 0:
        raise RuntimeError("device status %d during the swap benchmark" % int(status.item()))
    total_ms, moved = aggregate(t_out + t_in, 2.0 * bytes_one_way, world)
    gbs = lambda ms: bytes_one_way / (ms / 1e3) / 1e9
    # CPU baseline: the same block gather done on the host (numpy fancy indexing)
    hsrc = np.empty((2048, hkv * bs * d), dtype=np.float16)
    idx = rng.permutation(2048)[:1024]
    t0 = time.perf_counter()
    reps = 0
    while time.perf_counter() - t0 < 3.0:
        _ = hsrc[idx].copy()
        reps += 1
    cpu_gbs = reps * 1024 * hkv * bs * d * 2 / (time.perf_counter() - t0) / 1e9
    line = {
        "metric": "block swap GB/s (device cache <-> page-locked host, out + in)",
        "value": round(moved / (total_ms / 1e3) / 1e9, 2), "unit": "GB/s", "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": "swap_4096_blocks_of_10000_32kvh_bs16_d128_fp16", "blocks": n,
                   "bytes_each_way": bytes_one_way, "l2": "inputs larger than L2 (1.07 GB each way)",
                   "parallelism": "replicas" if world > 1 else "single"},
        "clocks": clk.summary(),
        "swap_out_gbs": round(gbs(t_out), 2), "swap_in_gbs": round(gbs(t_in), 2),
        "gpu_launches": 2 * steps,
        "roofline": {"bound": "link", "kernel": "swap_blocks_kernel", "achieved": round(gbs(t_out), 2),
                     "peak": C2C_GBS_PER_DIRECTION, "unit": "GB/s",
                     "frac": round(gbs(t_out) / C2C_GBS_PER_DIRECTION, 4),
                     "peak_kind": "of nominal (NVLink-C2C between the Grace host and the GPU: 900 GB/s both "
                                  "directions together, 450 GB/s each way)",
                     "swap_in_frac": round(gbs(t_in) / C2C_GBS_PER_DIRECTION, 4),
                     "d2h_copy_engine_gbs": round(gbs(t_d2h), 2), "h2d_copy_engine_gbs": round(gbs(t_h2d), 2),
                     "copy_engine_note": "one contiguous cudaMemcpyAsync of the same bytes each way (torch copy_), "
                                         "measured in the same run: context, not the peak",
                     "traffic": None},
        "cpu_baseline": {"value": round(cpu_gbs, 2), "unit": "GB/s", "cores": 1, "kind": "numpy_gather",
                         "sample": "numpy gather of 1024 of 2048 host blocks of 256 KiB, %d passes" % reps},
    }
    return line


# ---------------------------------------------------------------------------
def run_decode(args, workload, dev, rank, world, cpu_budget=10.0):
    """One decode workload's record (not printed)."""
    case, wname = build_workload(workload, dev, args.num_seqs, args.pool_blocks)
    # the long-context configuration states its partition (512 tokens)
    partition = args.partition_size or (512 if workload == "long" else 0)
    step = DecodeStep(case, dev, partition, wname)
    # the K/V a step reads, plus everything else it touches
    small = step.kv_bytes + case.q.numel() * case.q.element_size() * 2 < L2_BYTES
    flush = L2Flush(dev, small)
    total_ms, decode_ms, clocks = timed_decode(step, args.steps, args.warmup, world, flush)
    total_ms, kv_sum = aggregate(total_ms, float(step.kv_bytes) * args.steps, world)
    seqs_sum = aggregate(0.0, float(step.B) * args.steps, world)[1]
    ms_per_step = total_ms / args.steps
    value = kv_sum / (total_ms / 1e3) / 1e9
    e2e_ms, h2d, d2h = timed_e2e(step, args.steps, args.warmup, world)
    e2e_ms, kv_e2e = aggregate(e2e_ms, float(step.kv_bytes) * args.steps, world)
    hbm, _, _, peak_kind = measured_peaks()
    # the HBM roofline counts the distinct rows read (a prompt block shared by
    # a sampling group is read from DRAM once and re-read from L2); the
    # metric's own value stays on the logical bytes
    unique_bytes = case.unique_kv_bytes()
    achieved = unique_bytes / (decode_ms / 1e3) / 1e9
    achieved_logical = step.kv_bytes / (decode_ms / 1e3) / 1e9
    graph_ms = timed_graph(step, args.steps, flush) if small else None
    fused_ms = timed_append(step, args.steps, args.warmup, flush)
    plain = None
    if step.has_groups:
        # the same step with the plain decode (each member reads the shared
        # prompt blocks itself; the re-reads are L2 hits)
        p_total, p_decode, _ = timed_decode(step, args.steps, args.warmup, world, flush, attend=step.decode)
        p_total, p_sum = aggregate(p_total, float(step.kv_bytes) * args.steps, world)
        plain = {"ms_per_step": round(p_total / args.steps, 5), "value": round(p_sum / (p_total / 1e3) / 1e9, 2),
                 "unit": "GB/s", "kernel_achieved": round(unique_bytes / (p_decode / 1e3) / 1e9, 1),
                 "kernel_frac": round(unique_bytes / (p_decode / 1e3) / 1e9 / hbm, 4),
                 "note": "the same step with the attention through pa_decode (no shared-prefix pass); not in value"}
    # a configuration that states its partition: the same step with the
    # library's automatic choice beside it
    auto = None
    if partition:
        astep = DecodeStep(case, dev, 0, wname)
        if astep.P_eff != step.P_eff:
            a_total, a_decode, _ = timed_decode(astep, args.steps, args.warmup, world, flush)
            a_total, a_sum = aggregate(a_total, float(astep.kv_bytes) * args.steps, world)
            auto = {"partition_size": astep.P_eff, "ms_per_step": round(a_total / args.steps, 5),
                    "value": round(a_sum / (a_total / 1e3) / 1e9, 2), "unit": "GB/s",
                    "kernel_achieved": round(unique_bytes / (a_decode / 1e3) / 1e9, 1),
                    "kernel_frac": round(unique_bytes / (a_decode / 1e3) / 1e9 / hbm, 4),
                    "note": "the same step with partition_size 0 (pa_decode_partition_size); not in value"}
        del astep
    src_hash = kernel_source_hash()
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "storage_dtype": {0: "f16", 1: "bf16", 2: "e4m3"}[case.kv_dtype],
        "data": "synthetic",
        "config": {"workload": wname, "num_seqs": step.B, "num_heads": case.num_heads,
                   "num_kv_heads": case.num_kv_heads, "head_size": case.head_size, "block_size": case.block_size,
                   "num_blocks": case.num_blocks, "kv_bytes_per_step": step.kv_bytes,
                   "unique_kv_bytes_per_step": unique_bytes,
                   "partition_size": step.P_eff,
                   "l2": ("L2 flushed between timed steps (%.3f MB of K/V per step < 129 MB L2; each step "
                          "timed on its own)" % (step.kv_bytes / 1e6)) if small else
                         "inputs larger than L2 (%.2f GB of K/V read per step > 129 MB L2)" % (step.kv_bytes / 1e9),
                   "parallelism": "replicas" if world > 1 else "single"},
        "seqs_per_s_per_layer": round(seqs_sum / (total_ms / 1e3), 1),
        "hbm_frac_of_8000": round(value / world / 8000.0, 4),
        "hbm_frac_of_8000_distinct": round(value / world / 8000.0 * unique_bytes / step.kv_bytes, 4),
        "clocks": clocks,
        "e2e": {"value": round(kv_e2e / (e2e_ms / 1e3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms / args.steps, 5), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "pipeline": E2E_NOTE},
        "gpu_launches": step.launches_per_step * args.steps,
        "fused_append": {"ms_per_step": round(fused_ms, 5),
                         "value": round(step.kv_bytes / (fused_ms / 1e3) / 1e9, 2), "unit": "GB/s",
                         "note": "the same step (new token written, then attended) as one pa_decode_append launch; "
                                 "each step timed on its own"},
        "auto_partition": auto,
        "plain_decode": plain,
        "graph": None if graph_ms is None else {
            "us_per_step": round(graph_ms * 1e3, 2), "value": round(step.kv_bytes / (graph_ms / 1e3) / 1e9, 2),
            "unit": "GB/s", "note": "the same step captured once as a CUDA graph and replayed (not in value)"},
        "attention_call": "pa_decode_cascade" if step.has_groups else "pa_decode",
        "roofline": {"bound": "hbm",
                     "kernel": ("pa_decode_cascade (paged_decode_kernel in group mode + partition merge)"
                                if step.has_groups else "pa_decode (paged_decode_kernel + partition merge)"),
                     "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "peak_kind": "of %s" % peak_kind,
                     "bytes": "distinct K/V rows read (unique_kv_bytes_per_step)",
                     "achieved_logical": round(achieved_logical, 1),
                     "traffic": ncu_traffic(workload, src_hash), "decode_ms": round(decode_ms, 5),
                     "kernel_src": src_hash},
    }
    if small:
        line["us_per_step"] = round(ms_per_step * 1e3, 2)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case, cpu_budget)
    del step, case
    return line


SUB_KEYS = ("n_gpus", "steps", "warmup", "higher_is_better", "scaling", "vs_baseline", "data")


def run_ours(args):
    rank, local_rank, world = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    def one(workload, cpu_budget=10.0):
        if workload == "swap":
            return run_swap(args, dev, rank, world)
        if workload == "mixed":
            case, wname = build_workload("mixed", dev)
            line = run_prefill(args, case, wname, dev, rank, world, cpu_budget)
            del case
            return line
        return run_decode(args, workload, dev, rank, world, cpu_budget)

    if args.workload == "all":
        # the headline line (the MHA decode layer) carries every other
        # configuration's record under "configs"
        line = one("mha")
        configs = {}
        for w in ("tiny", "gqa", "long", "mixed"):
            torch.cuda.empty_cache()
            sub = one(w, cpu_budget=5.0)
            for k in SUB_KEYS:
                sub.pop(k, None)
            configs[w] = sub
        line["configs"] = configs
    else:
        line = one(args.workload)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def build_workload_name(name, groups=64):
    return "gqa_decode_%dseq_32q8kv_d128_bs16_bf16_lognormal1000_shared4_pool_cow" % (4 * groups)


def oracle_sampled_case(inp):
    """The parallel-sampling batch built on the host for the reference arm:
    the pool's reference model in the library's order of operations, then the
    oracle's cache write and block copy (no GPU involved)."""
    import oracle
    from oracle.pool_model import BlockPoolModel
    m = BlockPoolModel(inp.num_blocks, inp.block_size, inp.free_order.tolist())
    ps, gsl, pr = [], [], []
    gs = inp.group_size
    for g, (L, P) in enumerate(zip(inp.group_lens.tolist(), inp.prompt_lens.tolist())):
        m.add_seq(g * gs)
        ps += m.append(g * gs, P)[0]
        for k in range(1, gs):
            m.fork(g * gs, g * gs + k)
        for k in range(gs):
            s_, c_ = m.append(g * gs + k, L - P)
            gsl += s_
            pr += c_
    kc, vc = W.as_bits(inp.k_cache_init), W.as_bits(inp.v_cache_init)
    oracle.cache_write(kc, vc, W.BF16, W.as_bits(inp.prompt_k), W.as_bits(inp.prompt_v), W.BF16,
                       np.asarray(ps, np.int64))
    oracle.copy_blocks(kc, vc, W.BF16, np.asarray(pr, np.int32).reshape(-1, 2))
    oracle.cache_write(kc, vc, W.BF16, W.as_bits(inp.gen_k), W.as_bits(inp.gen_v), W.BF16, np.asarray(gsl, np.int64))
    table, lens = m.block_table(list(range(inp.num_seqs)), inp.max_blocks)
    as_t = lambda bits: torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    return W.PagedCase(q=inp.q, k_cache=as_t(kc), v_cache=as_t(vc), block_table=torch.tensor(table, dtype=torch.int32),
                       seq_lens=torch.tensor(lens, dtype=torch.int32), q_dtype=W.BF16, kv_dtype=W.BF16,
                       num_heads=inp.num_heads, num_kv_heads=inp.num_kv_heads, head_size=inp.head_size,
                       block_size=inp.block_size, scale=inp.scale)


def run_reference(args):
    """The CPU oracle on the host cores, each step a bounded sample."""
    rank, _, world = dist_env()
    if rank != 0:
        return
    if args.workload == "swap":
        # a block swap is a copy: the host-side reference gathers the same
        # blocks with numpy, host memory to host memory
        hkv, bs, d = 32, 16, 128
        rng = np.random.default_rng(778)
        src = np.empty((2048, hkv * bs * d), dtype=np.float16)
        idx = rng.permutation(2048)[:1024]
        for _ in range(args.warmup):
            src[idx].copy()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            src[idx].copy()
        dt = time.perf_counter() - t0
        value = args.steps * 1024 * hkv * bs * d * 2 / dt / 1e9
        print(json.dumps({
            "impl": "reference", "metric": "block swap GB/s (device cache <-> page-locked host, out + in)",
            "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": "swap_4096_blocks_of_10000_32kvh_bs16_d128_fp16"},
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": "numpy gather of 1024 of 2048 host blocks of 256 KiB per step"},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }), flush=True)
        return
    import oracle
    workload = "mha" if args.workload == "all" else args.workload  # the headline line's workload
    if workload == "gqa":
        case, wname = oracle_sampled_case(W.gqa_sampling_inputs(device="cpu")), build_workload_name("gqa")
    else:
        case, wname = build_workload(workload, "cpu")
    cores = os.cpu_count() or 1
    n = oracle.num_threads(cores)
    if workload == "mixed":
        kc, vc = W.as_bits(case.k_cache), W.as_bits(case.v_cache)
        sample = prefill_sample(case, rows_per_prefill=1, decode_every=12)
        flops = 4 * case.head_size * case.num_heads * sample[4]
        for _ in range(args.warmup):
            oracle_prefill_seconds(case, sample, n, kc, vc)
        spent = 0.0
        for _ in range(args.steps):
            spent += oracle_prefill_seconds(case, sample, n, kc, vc)
        value = flops * args.steps / spent / 1e12
        desc = ("oracle varlen prefill (fp64) over the last query row of each prefill sequence and every "
                "12th decode sequence (%.2f GFLOP) per step" % (flops / 1e9))
        print(json.dumps({
            "impl": "reference", "metric": "paged-attn varlen prefill TFLOP/s (causal, % of GB300 bf16 tensor peak)",
            "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(spent / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wname, "num_seqs": case.num_seqs, "sampled_rows": int(sample[2][-1])},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": n, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }), flush=True)
        return
    q_bits, kc, vc = W.as_bits(case.q), W.as_bits(case.k_cache), W.as_bits(case.v_cache)
    bt = case.block_table.numpy()
    lens = case.seq_lens.numpy()
    idx, sample_bytes = cpu_sample_indices(case, 3e8)
    for _ in range(args.warmup):
        oracle_decode_seconds(case, idx, n, q_bits, kc, vc, bt, lens)
    spent = 0.0
    for _ in range(args.steps):
        spent += oracle_decode_seconds(case, idx, n, q_bits, kc, vc, bt, lens)
    value = sample_bytes * args.steps / spent / 1e9
    sample = "oracle decode (fp64) over %d of %d sequences (%.1f MB of KV) per step" % (
        len(idx), case.num_seqs, sample_bytes / 1e6)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(spent / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wname, "num_seqs": case.num_seqs, "sampled_seqs": len(idx)},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": n, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["all", "mha", "gqa", "long", "tiny", "mixed", "swap"], default="all")
    ap.add_argument("--partition-size", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--num-seqs", type=int, default=None, help="sequences (smaller profiling cases)")
    ap.add_argument("--pool-blocks", type=int, default=None, help="mha workload: physical blocks in the pool")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
