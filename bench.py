#!/usr/bin/env python3
"""Benchmark of the paged-attention decode step on GB300.

Metric: paged decode attention KV-tokens/s (and HBM GB/s as a fraction of
the measured HBM peak) at 1 GPU.  Headline workload (default): the largest
single-GPU one, the bf16 decode batch of 256 sequences with the pages' skewed
length mix (70 % U[32,511], 25 % U[512,2047], 5 % U[2048,4095]), MHA 32 heads,
head_dim 128, 16-token blocks scattered through a pool sized to demand + 10 %,
one new token appended per sequence and step.  Every other workload of the
pages (the tiny fp32 case, the GQA-4 batch of 64, parallel sampling with
copy-on-write, and 4 x 128K-token contexts at block size 16 and 32) is
measured the same way in the same run and reported under `per_config`.

One step = the whole hot path for one decode iteration of the batch:
  a1 host allocator appends one token per sequence (slots, CoW pairs, tables)
  a2 copy-on-write block copy (only when the allocator emitted pairs)
  a3 slot-mapped append of the new K/V
  a4/a5 paged decode attention over len + 1 tokens (split, merged on the device)
`value` times a2-a5 on the device (CUDA events, inputs resident in HBM, L2
flushed between steps); the host allocator runs before the timed loop and
its time is reported separately.  `e2e` runs genuine decode steps through
the public API: host allocator, pinned host -> device copies of the step's
inputs, the kernels, and the device -> host copy of the output.

N > 1 (torchrun): every rank owns its own batch (weak scaling, no
data-path collective); the timed region is bracketed by barriers and the
max time over ranks is used.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "paged decode attention KV-tokens/s and HBM GB/s (% of GB300 roofline) at 1 GPU"
UNIT = "KV-tokens/s"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 512 << 20


# ---------------------------------------------------------------------------
# distributed plumbing (host-level only: barriers and the max of the times)
# ---------------------------------------------------------------------------
def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


def dist_init(world: int, backend: str):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def shard_lengths(global_lengths: np.ndarray, rank: int, world: int, per_rank: int) -> np.ndarray:
    """Sequences of this rank: a contiguous slice of the global draw (rank r owns r*per_rank ...)."""
    assert len(global_lengths) >= world * per_rank
    return np.asarray(global_lengths[rank * per_rank:(rank + 1) * per_rank], np.int32)


def reduce_max(x: float, dist, device) -> float:
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, dist, device) -> float:
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region (NVML through ctypes; nvidia-smi fallback)
# ---------------------------------------------------------------------------
REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
           0x80: "hw_power_brake_slowdown", 0x2: "applications_clocks_setting", 0x1: "gpu_idle"}


class ClockSampler:
    def __init__(self, cuda_index: int, period_s: float = 0.002):
        self.period = period_s
        self.samples = []  # (sm_mhz, reasons_mask)
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        self._handle = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit")
            handle = ctypes.c_void_p()
            bus = self._pci_bus_id(cuda_index)
            ok = bus is not None and nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(handle)) == 0
            if not ok and nv.nvmlDeviceGetHandleByIndex_v2(cuda_index, ctypes.byref(handle)) != 0:
                raise OSError("nvml handle")
            mx = ctypes.c_uint(0)
            if nv.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
            self._nvml, self._handle = nv, handle
        except OSError:
            self._nvml = None

    @staticmethod
    def _pci_bus_id(idx):
        try:
            import torch

            p = torch.cuda.get_device_properties(idx)
            return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
        except Exception:
            return None

    def _loop_nvml(self):
        nv, h = self._nvml, self._handle
        clk, rs = ctypes.c_uint(0), ctypes.c_ulonglong(0)
        get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and get_reasons(h, ctypes.byref(rs)) == 0:
                self.samples.append((int(clk.value), int(rs.value)))
            time.sleep(self.period)

    def start(self):
        if self._nvml is not None:
            self._thread = threading.Thread(target=self._loop_nvml, daemon=True)
            self._thread.start()

    def stop(self):
        self._stop.set()
        if self._thread:
            self._thread.join()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": "nvml" if self._nvml else "unavailable"}
        mhz = [s[0] for s in self.samples]
        mask = 0
        for _, r in self.samples:
            mask |= r
        reasons = [name for bit, name in sorted(REASONS.items()) if mask & bit and name != "gpu_idle"]
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(mhz), "source": "nvml"}


# ---------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------
WORKLOADS = {
    "tiny_f32": "fp32 decode of 4 sequences with lengths {5,17,33,48}, MHA 4 heads, d 64, 16-token blocks, 32-block pool",
    "gqa4_b64": "bf16 decode batch of 64 skew-mixed lengths, 32 query / 8 KV heads, d 128, 16-token blocks",
    "mha_b256_append": "bf16 decode batch of 256 skew-mixed lengths, MHA 32 heads, d 128, one appended token per step",
    "cow_sampling": "16 prompts of 1031 tokens forked into 8 samples each (refcount-shared blocks), tails U[0,256], "
                    "32 query / 8 KV heads, d 128",
    "long_context_bs16": "4 x 131072-token contexts, 64 query / 8 KV heads, d 128, 16-token blocks, 2048-token partitions",
    "long_context_bs32": "4 x 131072-token contexts, 64 query / 8 KV heads, d 128, 32-token blocks, 2048-token partitions",
}


def build_workload(name: str, rank: int, world: int, extra_steps: int):
    """The workload of this rank, with pool room for ``extra_steps`` more tokens per sequence."""
    import synth
    import synth.workloads as W

    if name not in WORKLOADS:
        raise SystemExit(f"unknown workload {name}; one of {sorted(WORKLOADS)}")
    seed_shift = 7919 * rank
    if name == "tiny_f32":
        base = W.tiny_fp32()
        demand = int(sum(-(-(int(x) + extra_steps) // base.block_size) for x in base.lengths))
        return W.scaled(base, num_blocks=max(base.num_blocks, demand), seed=base.seed + seed_shift)
    if name == "gqa4_b64":
        # every rank owns its own slice of one global length draw
        base = W.gqa4_b64()
        per_rank = base.num_seqs
        glob = synth.lengths_mix(synth.stream_seed(base.seed, W.TAG_LENGTHS), per_rank * world)
        lengths = shard_lengths(glob, rank, world, per_rank)
        demand = int(sum(-(-(int(x) + extra_steps) // base.block_size) for x in lengths))
        return W.scaled(base, lengths=lengths, num_blocks=int(math.ceil(1.1 * demand)), seed=base.seed + seed_shift)
    if name == "cow_sampling":
        base = W.cow_sampling()
        room = base.prompts * base.samples * (-(-extra_steps // base.block_size) + 1)
        return W.scaled(base, num_blocks=int(math.ceil(base.num_blocks + 1.1 * room)), seed=base.seed + seed_shift)
    base = W.mha_b256_append() if name == "mha_b256_append" else W.long_context(block_size=int(name[-2:]))
    demand = int(sum(-(-(int(x) + extra_steps) // base.block_size) for x in base.lengths))
    return W.scaled(base, num_blocks=int(math.ceil(1.1 * demand)), seed=base.seed + seed_shift)


def populate(alloc, w):
    """Build the workload's cache state through an allocator (ours or the oracle's model).

    Returns the ids of the decode batch's sequences, in batch order.  Parallel
    sampling forks every prompt into its samples, frees the prompt (its blocks
    stay shared by the samples), then appends the divergent tails one decode
    step at a time, which copies each shared partial prompt block on its first
    write.
    """
    if w.prompts:
        P, S, L = w.prompts, w.samples, w.prompt_len
        for p in range(P):
            alloc.create(p)
            alloc.append(p, L)
        sid = lambda p, s: P + p * S + s  # noqa: E731
        for p in range(P):
            for s in range(S):
                alloc.fork(p, sid(p, s))
            alloc.free_seq(p)
        tails = w.tails()
        for t in range(int(tails.max())):
            alloc.append_batch([sid(p, s) for p in range(P) for s in range(S) if tails[p * S + s] > t])
        return [sid(p, s) for p in range(P) for s in range(S)]
    for s, n in enumerate(w.lengths):
        alloc.create(s)
        alloc.append(s, int(n))
    return list(range(len(w.lengths)))


def decode_bytes(lens, w, kv_elem=None) -> int:
    """Algorithmic bytes of one decode launch: K and V of every token, tables, lengths, q and out."""
    e = w.elem_bytes
    kv = int(np.sum(lens, dtype=np.int64)) * w.num_kv_heads * w.head_dim * 2 * (kv_elem or e)
    tables = int(sum(-(-int(x) // w.block_size) for x in lens)) * 4
    qo = 2 * len(lens) * w.num_q_heads * w.head_dim * e
    return kv + tables + 4 * len(lens) + qo


def kernel_source_hash(csrc=None) -> str:
    """Hash of the code (comments and spacing dropped) the decode and merge kernels and their launch
    are built from, so that a recorded ncu figure survives edits to comments only."""
    import re
    h = hashlib.sha256()
    csrc = csrc or os.path.join(ROOT, "paged_kv_cache_280_gb300", "csrc")
    keep = ("pa_decode", "pa_device.cuh", "pa_internal.h", "pa_api.cu", "pa_plan.h")
    for f in sorted(x for x in os.listdir(csrc) if x.startswith(keep) and x.endswith((".cu", ".cuh", ".h"))):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            code = re.sub(r"/\*.*?\*/", " ", fh.read(), flags=re.S)
        code = re.sub(r"//[^\n]*", " ", code)
        h.update(f.encode() + " ".join(code.split()).encode())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# the headline: the largest single-GPU workload (2.66 GB of algorithmic bytes per decode)
DEFAULT_WORKLOAD = "mha_b256_append"
# every workload of the pages, in config order; the headline is one of them, the others go to per_config
PER_CONFIG = ["tiny_f32", "gqa4_b64", "mha_b256_append", "cow_sampling", "long_context_bs16", "long_context_bs32"]


def recorded_traffic(workload: str):
    """DRAM bytes per decode call (decode and merge kernels, bf16 pools) on this workload from the committed ncu
    summary, if it was taken on this kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"decode_{workload}_traffic.txt")
    try:
        with open(path) as f:
            kv = dict(line.split("=", 1) for line in f.read().split("\n") if "=" in line and not line.startswith("#"))
        if kv.get("kernel_source_hash", "").strip() == kernel_source_hash():
            return int(kv["dram_bytes_per_launch"].strip())
    except (OSError, ValueError, KeyError):
        pass
    return None


# ---------------------------------------------------------------------------
# CPU baseline: the oracle, as it stands, on the host cores
# ---------------------------------------------------------------------------
FP8_K_SCALE, FP8_V_SCALE = 1.0 / 64, 1.0 / 64  # N(0,1) draws over 1/64: codes up to about 300 of the 448 range


def fp8_codes(bf16_bits: np.ndarray, scale: float) -> np.ndarray:
    """E4M3 codes of bf16 values over a scale (synthetic pool contents, made with torch's conversion)."""
    import torch

    vals = torch.from_numpy(np.ascontiguousarray(bf16_bits).view(np.int16)).view(torch.bfloat16).float() / scale
    return vals.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def cpu_baseline(w, q, k_pool, v_pool, tables, lens, seconds: float, scales=None):
    """The oracle on the host cores over a bounded sample of the workload's sequences: rounds of as many
    sequences as there are threads (rotating through the batch) until `seconds` have passed, one round at
    least."""
    import oracle

    threads = os.cpu_count() or 1
    B = len(lens)
    chunk = max(1, min(B, threads))
    done_tokens, evals, rounds, start = 0, 0, 0, 0
    t0 = time.perf_counter()
    while True:
        seqs = sorted({(start + j) % B for j in range(chunk)})
        if scales:
            oracle.decode_attention_fp8(q, k_pool, v_pool, *scales, tables, lens, w.scale, seqs=seqs, threads=threads)
        else:
            oracle.decode_attention(q, k_pool, v_pool, tables, lens, w.scale, seqs=seqs, threads=threads)
        done_tokens += int(sum(int(lens[s]) for s in seqs))
        evals += len(seqs)
        rounds += 1
        start += chunk
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": done_tokens / dt, "unit": UNIT, "cores": min(threads, chunk), "kind": "oracle",
            "sample": f"fp64 C oracle, {rounds} round(s) of {chunk} of the {B} sequences (rotating), {evals} "
                      f"sequence evaluations in {dt:.1f} s, one thread per sequence"}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
class DecodeSetup:
    """One workload's decode step, device-resident: pools, the step's allocator outputs, q, out, workspace."""

    def __init__(self, name, args, rank, world, dev, pa, e2e_steps):
        import torch

        self.name, self.pa, self.dev = name, pa, dev
        self.w = w = build_workload(name, rank, world, extra_steps=1 + e2e_steps + 2)
        self.fp8 = fp8 = args.kv == "fp8"
        self.Hq, self.Hkv, self.D, self.bs, self.PT = w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, w.partition_tokens
        self.lib = pa.Allocator(w.num_blocks, self.bs, free_order=w.free_order())
        self.ids = populate(self.lib, w)
        self.B = B = len(self.ids)
        self.max_blocks = int(-(-(max(self.lib.length(s) for s in self.ids) + 2 + e2e_steps) // self.bs))
        self.k_host, self.v_host = w.pool_values("k"), w.pool_values("v")
        self.KS, self.VS = FP8_K_SCALE, FP8_V_SCALE
        if fp8:
            # FP8 pools: E4M3 codes of the same N(0,1) draws over the pool scales (input data, made on the host)
            self.k_host, self.v_host = fp8_codes(self.k_host, self.KS), fp8_codes(self.v_host, self.VS)
            self.dk, self.dv = torch.from_numpy(self.k_host).to(dev), torch.from_numpy(self.v_host).to(dev)
        else:
            self.dk, self.dv = self.to_dev(self.k_host), self.to_dev(self.v_host)
        # ---- a1 once: the step's allocator outputs become device-resident inputs ----
        t_alloc = time.perf_counter()
        slots, pairs = self.lib.append_batch(self.ids)
        self.tables, self.lens = self.lib.export_tables(self.ids, self.max_blocks)
        self.host_alloc_us = (time.perf_counter() - t_alloc) * 1e6
        self.q = w.queries(step=1)
        k_new, v_new = w.new_tokens("k", B, step=1), w.new_tokens("v", B, step=1)
        self.d_q, self.d_kn, self.d_vn = self.to_dev(self.q), self.to_dev(k_new), self.to_dev(v_new)
        self.d_slots, self.d_tables, self.d_lens = self.to_dev(slots), self.to_dev(self.tables), self.to_dev(self.lens)
        self.d_pairs = self.to_dev(pairs) if len(pairs) else None
        # kernels of one step: (CoW copy,) append, decode (and the merge kernel, when the call uses it)
        dt = pa.PA_FP8_E4M3 if self.fp8 else (pa.PA_F32 if w.dtype == "f32" else pa.PA_BF16)
        self.decode_kernels = pa.pa_decode_kernels_per_call(B, self.Hq, self.Hkv, self.D, self.bs, self.max_blocks,
                                                            self.PT, dt)
        self.launches_per_step = 1 + self.decode_kernels + (1 if self.d_pairs is not None else 0)
        self.out = torch.empty_like(self.d_q)
        self.ws = torch.zeros(pa.pa_decode_workspace_bytes(B, self.Hq, self.Hkv, self.D), dtype=torch.uint8, device=dev)
        self.max_len = int(self.lens.max())
        # the host's work plan of the decode call (built from the allocator's tables and lengths, uploaded
        # with them), unless --no-plan
        self.dtype_code = dt
        self.d_plan = None
        if not getattr(args, "no_plan", False):
            self.d_plan = self.to_dev(self.build_plan(self.tables, self.lens, self.max_len))

    def build_plan(self, tables, lens, max_len, out=None):
        return self.pa.pa_decode_build_plan(tables, lens, max_len, self.Hq, self.Hkv, self.D, self.bs, self.PT,
                                            self.dtype_code, out=out)

    def to_dev(self, a):
        import torch

        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(self.dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(self.dev)

    def append(self, kn_, vn_, slots_, **kw):
        if self.fp8:
            self.pa.pa_reshape_and_cache_fp8(kn_, vn_, self.dk, self.dv, slots_, self.KS, self.VS, **kw)
        else:
            self.pa.pa_reshape_and_cache(kn_, vn_, self.dk, self.dv, slots_, **kw)

    def attend(self, q_, tables_, lens_, max_len_, **kw):
        kw.setdefault("plan", self.d_plan)
        if self.fp8:
            self.pa.pa_decode_attention_fp8(self.out, q_, self.dk, self.dv, self.KS, self.VS, tables_, lens_, max_len_,
                                            self.w.scale, self.ws, partition_tokens=self.PT, **kw)
        else:
            self.pa.pa_decode_attention(self.out, q_, self.dk, self.dv, tables_, lens_, max_len_, self.w.scale, self.ws,
                                        partition_tokens=self.PT, **kw)

    def step(self, stream):
        """a2 (when the allocator emitted copy-on-write pairs) and a3."""
        st = self.ws[:4].view(__import__("torch").int32)
        if self.d_pairs is not None:
            self.pa.pa_copy_blocks(self.dk, self.dv, self.d_pairs, status=st, stream=stream)
        self.append(self.d_kn, self.d_vn, self.d_slots, status=st, stream=stream)

    def decode(self, stream):
        """a4 + a5: the decode call (the decode kernel, and the merge kernel when the call uses one)."""
        self.attend(self.d_q, self.d_tables, self.d_lens, self.max_len, stream=stream)

    def time_steps(self, K, Wm, flush_l2, stream, dist, on_timed=None):
        """W untimed steps, then K timed steps (events at their ends only) and K decode calls timed alone.

        An event between the append and the decode would keep the decode from starting its prologue while
        the append runs (it is launched as the append's programmatic dependent), so the steps carry events
        at their two ends only; the decode call alone is timed in a second loop of K, for the roofline."""
        import torch

        for _ in range(Wm):
            flush_l2()
            self.step(stream)
            self.decode(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        dev_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        if on_timed:
            on_timed(True)
        torch.cuda.synchronize()
        for i in range(K):
            flush_l2()
            ev[i][0].record(stream)
            self.step(stream)
            self.decode(stream)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        for i in range(K):
            flush_l2()
            self.step(stream)
            dev_ev[i][0].record(stream)
            self.decode(stream)
            dev_ev[i][1].record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        if on_timed:
            on_timed(False)
        status = int(self.ws[:4].view(torch.int32).item())
        if status:
            raise SystemExit(f"{self.name}: device status word {status:#x}")
        return [a.elapsed_time(b) for a, b in ev], [a.elapsed_time(b) for a, b in dev_ev]

    def bytes_and_unique(self):
        elem = 1 if self.fp8 else self.w.elem_bytes
        dbytes = decode_bytes(self.lens, self.w, kv_elem=elem)
        # KV bytes of the distinct physical blocks the step reads (below the per-sequence
        # bytes when sequences share prefix blocks, which L2 then serves more than once)
        used = [self.tables[i, : -(-int(n) // self.bs)] for i, n in enumerate(self.lens)]
        unique_kv = int(np.unique(np.concatenate(used)).size) * self.bs * self.Hkv * self.D * 2 * elem if self.B else 0
        return dbytes, unique_kv

    def summary(self, step_ms, dec_ms, peak):
        """Per-config figures: decode call time (median, mean), algorithmic GB/s and its fraction of the peak."""
        dbytes, unique_kv = self.bytes_and_unique()
        mean_s = statistics.mean(dec_ms) / 1e3
        tokens = int(np.sum(self.lens, dtype=np.int64))
        ctas, stages, smem, mma = self.pa.pa_decode_launch_info(self.B, self.Hq, self.Hkv, self.D, self.bs, self.max_blocks,
                                                                self.pa.PA_FP8_E4M3 if self.fp8 else
                                                                (self.pa.PA_F32 if self.w.dtype == "f32" else self.pa.PA_BF16),
                                                                partition_tokens=self.PT)
        d = {
            "workload": self.w.name + ("_fp8kv" if self.fp8 else ""), "dtype": self.w.dtype,
            "kv_tokens_per_step": tokens, "decode_bytes_per_step": dbytes,
            "step_ms_mean": statistics.mean(step_ms), "value_kv_tokens_per_s": tokens * len(step_ms) / (sum(step_ms) / 1e3),
            "decode_us_median": 1e3 * statistics.median(dec_ms), "decode_us_mean": 1e3 * statistics.mean(dec_ms),
            "decode_us_min": 1e3 * min(dec_ms), "decode_gbs": dbytes / mean_s / 1e9,
            "frac_of_measured_hbm": dbytes / mean_s / 1e9 / peak, "decode_ctas": ctas, "stages": stages,
            "path": "mma.sync" if mma else "fma", "partition_tokens": self.PT, "steps": len(step_ms),
            "launches_per_step": self.launches_per_step,
        }
        if self.w.prompts:  # shared prompt blocks: L2 serves them more than once
            d["unique_block_kv_bytes_per_step"] = unique_kv
            d["unique_block_gbs"] = unique_kv / mean_s / 1e9
        return d


def run_ours(args, rank, world, local_rank):
    import torch

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = dist_init(world, "nccl")
    import paged_kv_cache_280_gb300 as pa

    K, Wm = args.steps, args.warmup
    K_e2e = args.e2e_steps
    pa.pa_debug_set_merge_mode(args.merge_mode)
    pa.pa_decode_set_ctas_per_sm(args.ctas_per_sm)
    pa.pa_debug_set_seg_units(args.seg_units)
    pa.pa_debug_set_wave_skew(args.wave_skew)
    S = DecodeSetup(args.workload, args, rank, world, dev, pa, K_e2e)
    w, B, Hq, Hkv, D, bs = S.w, S.B, S.Hq, S.Hkv, S.D, S.bs
    fp8, ids, lib, max_blocks, out = S.fp8, S.ids, S.lib, S.max_blocks, S.out
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def flush_l2():
        # Write a buffer 4x the L2, then read half of it back: L2 ends up holding
        # only clean lines of the read, none of the step's inputs, so the step
        # neither hits in L2 nor pays for another kernel's dirty write-backs.
        flush.zero_()
        flush[: L2_FLUSH_BYTES // 2].view(torch.int32).sum()

    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local_rank)
    step_ms, dec_ms = S.time_steps(K, Wm, flush_l2, stream, dist,
                                   on_timed=lambda on: clocks.start() if on else clocks.stop())
    total_s = reduce_max(sum(step_ms) / 1e3, dist, dev)
    tokens_step = int(np.sum(S.lens, dtype=np.int64))
    all_tokens = reduce_sum(float(tokens_step * K), dist, dev)
    value = all_tokens / total_s
    dbytes, unique_kv = S.bytes_and_unique()
    dec_mean_s = statistics.mean(dec_ms) / 1e3
    peak, peak_kind = measured_peaks()
    achieved = dbytes / dec_mean_s / 1e9
    ctas, stages, smem, mma = pa.pa_decode_launch_info(B, Hq, Hkv, D, bs, max_blocks,
                                                       pa.PA_FP8_E4M3 if fp8 else
                                                       (pa.PA_F32 if w.dtype == "f32" else pa.PA_BF16),
                                                       partition_tokens=S.PT)

    # ---- e2e: genuine decode steps through the public API with host buffers ----
    # Each step's inputs travel in one pinned staging buffer, copied to the device
    # with one H2D copy: q, k_new, v_new (produced upstream, filled before the
    # loop), then the allocator's slots, CoW pairs, block tables and lengths,
    # which the allocator writes in place during the step.
    e = w.elem_bytes
    tdt, hdt = (torch.float32, torch.int32) if e == 4 else (torch.bfloat16, torch.int16)
    regions = [("q", B * Hq * D * e), ("kn", B * Hkv * D * e), ("vn", B * Hkv * D * e), ("slots", B * 8),
               ("pairs", B * 2 * 4), ("tables", B * max_blocks * 4), ("lens", B * 4)]
    cap_len = max_blocks * bs  # a length bound every step's tables respect
    use_plan = S.d_plan is not None
    if use_plan:  # the host's work plan of each step's decode call travels with its tables
        regions.append(("plan", pa.pa_decode_plan_bytes(B, Hq, Hkv, D, bs, max_blocks, cap_len, S.PT, S.dtype_code)))
    offs, pos = {}, 0
    for name, n in regions:
        offs[name] = (pos, n)
        pos += -(-n // 256) * 256
    stage_bytes = pos

    def region(buf, name, dtype, shape):
        o, n = offs[name]
        return buf[o:o + n].view(dtype).view(shape)

    # Two pinned staging buffers, used in turn: the allocator fills one while the GPU copies the
    # other.  Their q and new K/V (made upstream) alternate between two draws.
    n_stage = min(2, K_e2e)
    host_stage = [torch.empty(stage_bytes, dtype=torch.uint8).pin_memory() for _ in range(n_stage)]
    for s, hb in enumerate(host_stage):
        for name, src in (("q", w.queries(step=2 + s)), ("kn", w.new_tokens("k", B, step=2 + s)),
                          ("vn", w.new_tokens("v", B, step=2 + s))):
            o, n = offs[name]
            hb.numpy()[o:o + n] = np.ascontiguousarray(src).view(np.uint8).reshape(-1)
    dev_stage = torch.empty(stage_bytes, dtype=torch.uint8, device=dev)
    e_q = region(dev_stage, "q", tdt, (B, Hq, D))
    e_kn = region(dev_stage, "kn", tdt, (B, Hkv, D))
    e_vn = region(dev_stage, "vn", tdt, (B, Hkv, D))
    e_slots = region(dev_stage, "slots", torch.int64, (B,))
    e_pairs = region(dev_stage, "pairs", torch.int32, (B, 2))
    e_tables = region(dev_stage, "tables", torch.int32, (B, max_blocks))
    e_lens = region(dev_stage, "lens", torch.int32, (B,))
    e_plan = region(dev_stage, "plan", torch.int32, (-1,)) if use_plan else None
    h_out = torch.empty((B, Hq, D), dtype=hdt).pin_memory()
    ids_arr = np.asarray(ids, np.int64)

    def device_step(hb, max_len_, st):
        dev_stage.copy_(hb, non_blocking=True)
        S.append(e_kn, e_vn, e_slots, stream=st)
        S.attend(e_q, e_tables, e_lens, max_len_, stream=st, plan=e_plan)
        h_out.copy_(out.view(hdt), non_blocking=True)

    graphs = []
    if not args.e2e_eager:
        # One CUDA graph per staging buffer: its H2D copy, the append, the decode and the D2H of the
        # output replay as one launch.  The library's per-call setup is cached by the timed loop above.
        for hb in host_stage:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                device_step(hb, cap_len, torch.cuda.current_stream())
            graphs.append(g)
        torch.cuda.synchronize()
    # numpy views of each staging buffer's allocator regions, made once
    host_views = [(region(hb, "slots", torch.int64, (B,)).numpy(), region(hb, "pairs", torch.int32, (B, 2)).numpy(),
                   region(hb, "tables", torch.int32, (B, max_blocks)).numpy(), region(hb, "lens", torch.int32, (B,)).numpy(),
                   region(hb, "plan", torch.int32, (-1,)).numpy() if use_plan else None)
                  for hb in host_stage]

    host_us = []

    def host_prepare(s):
        # the allocator's step: new slots (and CoW pairs), block tables and lengths,
        # written in place into staging buffer s % 2, and the decode call's plan
        t_host = time.perf_counter()
        h_slots, h_pairs, h_tables, h_lens, h_plan = host_views[s % n_stage]
        _, pr = lib.append_batch(ids_arr, slots_out=h_slots, pairs_out=h_pairs)
        lib.export_tables(ids_arr, max_blocks, tables_out=h_tables, lens_out=h_lens)
        if use_plan:
            S.build_plan(h_tables, h_lens, cap_len, out=h_plan)
        host_us.append((time.perf_counter() - t_host) * 1e6)
        return pr, int(h_lens.sum(dtype=np.int64))

    def gpu_step(s, pr):
        if graphs and not len(pr):
            graphs[s % n_stage].replay()
        else:  # copy-on-write pairs go between the H2D copy and the append: launched one by one
            dev_stage.copy_(host_stage[s % n_stage], non_blocking=True)
            if len(pr):
                pa.pa_copy_blocks(S.dk, S.dv, e_pairs[: len(pr)], stream=stream)
            S.append(e_kn, e_vn, e_slots, stream=stream)
            S.attend(e_q, e_tables, e_lens, cap_len, stream=stream, plan=e_plan)
            h_out.copy_(out.view(hdt), non_blocking=True)

    # The allocator runs one step ahead of the GPU, as a serving loop's scheduler does: step s+1's
    # slots and tables are written into their own staging buffer while the GPU runs step s.  Every
    # step still copies its inputs host to device and reads its output back before the next step
    # is launched.  No L2 flush runs inside this loop: the KV a step reads is larger than L2 and
    # is loaded with an evict-first policy.
    e2e_tokens, h2d, d2h, launches = 0, 0, 0, 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    if K_e2e:
        pr, toks = host_prepare(0)
    for s in range(K_e2e):
        gpu_step(s, pr)
        e2e_tokens += toks
        h2d += stage_bytes
        d2h += h_out.numel() * e
        launches += 3 + (1 if len(pr) else 0)
        if s + 1 < K_e2e:
            pr, toks = host_prepare(s + 1)
        stream.synchronize()  # step s's output is on the host
    e2e_s = time.perf_counter() - t0
    e2e_total = reduce_max(e2e_s, dist, dev)
    e2e_value = reduce_sum(float(e2e_tokens), dist, dev) / e2e_total if K_e2e else None

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": total_s * 1e3 / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8_e4m3 kv, bf16 q/out" if fp8 else w.dtype,
        "data": f"synthetic, seeded: {WORKLOADS[args.workload]}; blocks scattered by a seeded free-list order",
        "config": {
            "workload": (w.name + ("_fp8kv" if fp8 else "")) if world == 1 else f"{w.name} per rank",
            "num_seqs_per_gpu": B, "num_q_heads": Hq,
            "num_kv_heads": Hkv, "head_dim": D, "block_size": bs, "kv_tokens_per_step": tokens_step,
            "decode_bytes_per_step": dbytes, "unique_block_kv_bytes_per_step": unique_kv, "pool_blocks": w.num_blocks,
            "timing": "steps (append + decode call) timed with events at their ends only; the decode call "
                      "(decode kernel, and merge kernel when used) timed alone in a second loop of as many steps",
            "l2": f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MiB write, then a {L2_FLUSH_BYTES >> 21} MiB read "
                  "so that no dirty line is left; untimed)",
            "host_alloc_us_first_call": round(S.host_alloc_us, 1),
            "host_prepare_us_median": round(statistics.median(host_us), 1) if host_us else None,
            "host_prepare": "the allocator's step (slots, CoW pairs, block tables, lengths) and the decode plan, "
                            "written into pinned staging; median over the end-to-end steps",
            "decode_ctas": ctas, "stages": stages,
            "smem_bytes": smem, "path": "mma.sync" if mma else "fma", "partition_tokens": S.PT,
            "kv_dtype": "fp8_e4m3" if fp8 else "bf16", **({"k_scale": S.KS, "v_scale": S.VS} if fp8 else {}),
            "decode_ms_median": statistics.median(dec_ms), "decode_ms_min": min(dec_ms),
            "step_gbs": (dbytes + 4 * B * Hkv * D * 2) / (total_s / K) / 1e9,
        },
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback",
                     "kernel": "pa_decode_attention (" + ("decode kernel, merging split segments itself)"
                                                          if S.decode_kernels == 1 else "decode kernel, then merge kernel)"),
                     "traffic": None if fp8 else recorded_traffic(args.workload)},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d // max(1, K_e2e),
                "d2h_bytes_per_step": d2h // max(1, K_e2e), "steps": K_e2e,
                "includes": "host allocator" + (" and decode plan" if use_plan else "") + " writing into pinned "
                            "staging one step ahead of the GPU, one H2D of q/k_new/v_new/slots/pairs/tables/lens"
                            + ("/plan" if use_plan else "") + ", kernels, D2H of out; no L2 flush inside the loop "
                            "(the KV read per step is larger than L2 and loaded evict-first)",
                "launch": "eager" if args.e2e_eager else "one CUDA graph per staging buffer (H2D, append, decode (+ merge), D2H)"},
        "gpu_launches": K * S.launches_per_step,
        "clocks": clocks.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, S.q, S.k_host, S.v_host, S.tables, S.lens, args.cpu_seconds,
                                            scales=(S.KS, S.VS) if fp8 else None)
    # The other workloads of the pages (every config that is not the headline), each measured the same way
    # on this machine in this run, with its own bounded CPU baseline.  Single-GPU runs only.
    if world == 1 and not args.no_per_config:
        del S, dev_stage, graphs, host_stage
        torch.cuda.empty_cache()
        per = {}
        all_samples = []
        for name in PER_CONFIG:
            if name == args.workload or (fp8 and name == "tiny_f32"):
                continue
            C = DecodeSetup(name, args, 0, 1, dev, pa, 0)
            cs = ClockSampler(local_rank)
            sm, dm = C.time_steps(args.per_config_steps, 3, flush_l2, stream, None,
                                  on_timed=lambda on, cs=cs: cs.start() if on else cs.stop())
            d = C.summary(sm, dm, peak)
            d["clocks"] = cs.summary()
            all_samples += cs.samples
            d["traffic"] = None if fp8 else recorded_traffic(name)
            if not args.no_cpu_baseline:
                d["cpu_baseline"] = cpu_baseline(C.w, C.q, C.k_host, C.v_host, C.tables, C.lens,
                                                 args.per_config_cpu_seconds, scales=(C.KS, C.VS) if fp8 else None)
            per[name] = d
            del C
            torch.cuda.empty_cache()
        line["per_config"] = per
        agg = ClockSampler.__new__(ClockSampler)
        agg.samples, agg.max_mhz, agg._nvml = all_samples, line["clocks"].get("sm_max_mhz"), True
        line["per_config_clocks"] = agg.summary()
        line["gpu_launches_per_config"] = {k: v["steps"] * v["launches_per_step"] for k, v in per.items()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# prefill path: prompt prefill of the parallel-sampling workload
# ---------------------------------------------------------------------------
PREFILL_METRIC = "paged prefill attention prompt-tokens/s and TFLOP/s (% of GB300 bf16 tensor roofline) at 1 GPU"
PREFILL_UNIT = "prompt-tokens/s"


def measured_tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def prefill_setup(rank: int, prompts: int):
    """Prompts of the parallel-sampling workload, each prefilled as one chunk."""
    import synth
    import synth.workloads as W

    base = W.cow_sampling()
    P, L, bs = min(prompts, base.prompts), base.prompt_len, base.block_size
    nb = int(math.ceil(1.1 * P * -(-L // bs)))
    return W.scaled(base, prompts=P, num_blocks=nb, seed=base.seed + 7919 * rank), P, L


def prefill_flops(L: int, P: int, hq: int, d: int, chunk: int = 0) -> float:
    """Causal attention of the last ``chunk`` tokens (all L by default) of P prompts of L tokens:
    4 d Hq (p + 1) per chunk token at position p (QK^T and PV)."""
    chunk = chunk or L
    return 4.0 * d * hq * P * sum(L - chunk + i + 1 for i in range(chunk))


def run_prefill(args, rank, world, local_rank):
    import torch
    import synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = dist_init(world, "nccl")
    import paged_kv_cache_280_gb300 as pa

    K, Wm = args.steps, args.warmup
    K_e2e = min(K, args.e2e_steps)
    w, P, L = prefill_setup(rank, args.prompts)
    Hq, Hkv, D, bs = w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size
    lib = pa.Allocator(w.num_blocks, bs, free_order=w.free_order())
    slots = []
    if args.prefix_cached:
        # The prompts share their first L - 7 tokens (a system prompt).  An earlier request
        # computed that prefix and registered it (untimed): each prompt now reuses those
        # blocks and computes only its own 7-token tail, attending to all L tokens.
        chunk = 7
        shared = [10_000 + t for t in range(L - chunk)]
        toks = [shared + [100 * p_ + t for t in range(chunk)] for p_ in range(P)]
        lib.create(1 << 40)
        lib.append(1 << 40, L)
        lib.cache_prefix(1 << 40, toks[0])
        lib.free_seq(1 << 40)  # the prefix blocks stay cached
        for p_ in range(P):
            if lib.create_cached(p_, toks[p_]) != L - chunk:
                raise SystemExit("prefix cache missed")
            slots.append(lib.append(p_, chunk)[0])
    else:
        chunk = L
        for p_ in range(P):
            lib.create(p_)
            slots.append(lib.append(p_, L)[0])
    T = P * chunk
    slots = np.concatenate(slots)
    max_blocks = -(-L // bs)
    tables, lens = lib.export_tables(range(P), max_blocks)
    cu = np.arange(0, T + 1, chunk, dtype=np.int32)
    q = synth.normal(synth.stream_seed(w.seed, 4242), T * Hq * D, "bf16").reshape(T, Hq, D)
    kn, vn = w.prompt_tokens("k")[:T], w.prompt_tokens("v")[:T]

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    k_host, v_host = w.pool_values("k"), w.pool_values("v")
    dk, dv = to_dev(k_host), to_dev(v_host)
    d_q, d_kn, d_vn = to_dev(q), to_dev(kn), to_dev(vn)
    d_slots, d_tables, d_lens, d_cu = to_dev(slots), to_dev(tables), to_dev(lens), to_dev(cu)
    out = torch.empty_like(d_q)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def flush_l2():
        flush.zero_()
        flush[: L2_FLUSH_BYTES // 2].view(torch.int32).sum()

    def append(kk, vv, ss):
        pa.pa_reshape_and_cache(kk, vv, dk, dv, ss, status=status, stream=stream)

    def prefill(qq, tt, ll, cc):
        pa.pa_prefill_attention(out, qq, dk, dv, tt, ll, cc, chunk, w.scale, status=status, stream=stream)

    for _ in range(Wm):
        flush_l2()
        append(d_kn, d_vn, d_slots)
        prefill(d_q, d_tables, d_lens, d_cu)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(K)]
    clocks = ClockSampler(local_rank)
    clocks.start()
    torch.cuda.synchronize()
    for i in range(K):
        flush_l2()
        ev[i][0].record(stream)
        append(d_kn, d_vn, d_slots)
        ev[i][1].record(stream)
        prefill(d_q, d_tables, d_lens, d_cu)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks.stop()
    if status.item():
        raise SystemExit(f"device status word {int(status.item()):#x}")
    step_ms = [a.elapsed_time(c) for a, b, c in ev]
    pf_ms = [b.elapsed_time(c) for a, b, c in ev]
    total_s = reduce_max(sum(step_ms) / 1e3, dist, dev)
    value = reduce_sum(float(P * L * K), dist, dev) / total_s  # prompt tokens made ready (cached ones included)
    flops = prefill_flops(L, P, Hq, D, chunk)
    peak, peak_kind = measured_tensor_peak()
    achieved = flops / (statistics.mean(pf_ms) / 1e3) / 1e12

    # e2e: one pinned staging buffer per step (q, new K/V, slots, tables, lengths, chunk offsets), one H2D,
    # the two kernels, and the D2H of the output
    regions = [("q", T * Hq * D * 2), ("kn", T * Hkv * D * 2), ("vn", T * Hkv * D * 2), ("slots", T * 8),
               ("tables", P * max_blocks * 4), ("lens", P * 4), ("cu", (P + 1) * 4)]
    offs, pos = {}, 0
    for name, n in regions:
        offs[name] = (pos, n)
        pos += -(-n // 256) * 256
    host_stage = torch.empty(pos, dtype=torch.uint8).pin_memory()
    for name, src in (("q", q), ("kn", kn), ("vn", vn), ("slots", slots), ("tables", tables), ("lens", lens),
                      ("cu", cu)):
        o, n = offs[name]
        host_stage.numpy()[o:o + n] = np.ascontiguousarray(src).view(np.uint8).reshape(-1)
    dev_stage = torch.empty(pos, dtype=torch.uint8, device=dev)

    def region(name, dtype, shape):
        o, n = offs[name]
        return dev_stage[o:o + n].view(dtype).view(shape)

    e_q, e_kn, e_vn = region("q", torch.bfloat16, (T, Hq, D)), region("kn", torch.bfloat16, (T, Hkv, D)), \
        region("vn", torch.bfloat16, (T, Hkv, D))
    e_slots, e_tables = region("slots", torch.int64, (T,)), region("tables", torch.int32, (P, max_blocks))
    e_lens, e_cu = region("lens", torch.int32, (P,)), region("cu", torch.int32, (P + 1,))
    h_out = torch.empty((T, Hq, D), dtype=torch.int16).pin_memory()
    e2e_s = 0.0
    for _ in range(K_e2e):
        flush_l2()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        dev_stage.copy_(host_stage, non_blocking=True)
        append(e_kn, e_vn, e_slots)
        prefill(e_q, e_tables, e_lens, e_cu)
        h_out.copy_(out.view(torch.int16), non_blocking=True)
        stream.synchronize()
        e2e_s += time.perf_counter() - t0
    e2e_total = reduce_max(e2e_s, dist, dev)
    e2e_value = reduce_sum(float(P * L * K_e2e), dist, dev) / e2e_total if K_e2e else None

    line = {
        "metric": PREFILL_METRIC, "value": value, "unit": PREFILL_UNIT, "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": total_s * 1e3 / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": f"synthetic, seeded: {P} prompts of {L} tokens (the parallel-sampling workload's "
                                 f"prompts), 32 query / 8 KV heads, d 128, 16-token blocks scattered",
        "config": {"workload": f"prefill_p{P}_len{L}_hq{Hq}_hkv{Hkv}_d{D}_bs{bs}_bf16"
                               + ("_prefix_cached" if args.prefix_cached else ""), "prompts": P,
                   "prompt_len": L, "computed_tokens_per_prompt": chunk, "cached_tokens_per_prompt": L - chunk,
                   "num_q_heads": Hq, "num_kv_heads": Hkv, "head_dim": D, "block_size": bs,
                   "flops_per_step": flops, "l2": "flushed between timed steps (512 MiB write, then a 256 MiB read)",
                   "prefill_ms_median": statistics.median(pf_ms), "prefill_ms_min": min(pf_ms),
                   "path": "tcgen05.mma (TMEM accumulators, P in TMEM), TMA ring"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                     "peak_source": peak_kind, "kernel": "pa_prefill_attention (prefill_kernel)", "traffic": None},
        "e2e": {"value": e2e_value, "unit": PREFILL_UNIT, "h2d_bytes_per_step": pos,
                "d2h_bytes_per_step": h_out.numel() * 2, "steps": K_e2e,
                "includes": "one H2D of the pinned staging (q, new K/V, slots, tables, lengths, offsets), the append "
                            "and prefill kernels, D2H of out"},
        "gpu_launches": 2 * K,
        "clocks": clocks.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = prefill_cpu_baseline(w, q, k_host, v_host, kn, vn, slots, tables, lens, L, P, chunk,
                                                    args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def prefill_cpu_baseline(w, q, k_pool, v_pool, kn, vn, slots, tables, lens, L, P, chunk, seconds):
    """The oracle's prefill of the same chunks (one prompt per host thread at a time), bounded by ``seconds``."""
    import oracle

    k_pool, v_pool = k_pool.copy(), v_pool.copy()
    oracle.reshape_and_cache(kn, vn, k_pool, v_pool, slots)
    threads = os.cpu_count() or 1
    cu = np.arange(0, P * chunk + 1, chunk, dtype=np.int32)
    done, t0 = 0, time.perf_counter()
    while done < P:
        seqs = list(range(done, min(P, done + threads)))
        oracle.prefill_attention(q, k_pool, v_pool, tables, lens, cu, w.scale, seqs=seqs, threads=threads)
        done += len(seqs)
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": done * L / dt, "unit": PREFILL_UNIT, "cores": threads, "kind": "oracle",
            "sample": f"fp64 C oracle prefill of {done} of the {P} prompts ({chunk} computed tokens each, "
                      f"{dt:.1f} s), one prompt per thread"}


# ---------------------------------------------------------------------------
# swap path: preempt the whole decode batch to pinned host memory and back
# ---------------------------------------------------------------------------
SWAP_METRIC = "paged KV swap-out + swap-in GB/s (% of the pinned-memcpy link rate) at 1 GPU"


def run_swap(args, rank, world, local_rank):
    import torch

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = dist_init(world, "nccl")
    import paged_kv_cache_280_gb300 as pa

    K, Wm = args.steps, args.warmup
    w = build_workload("gqa4_b64", rank, world, extra_steps=0)
    Hkv, D, bs = w.num_kv_heads, w.head_dim, w.block_size
    lib = pa.Allocator(w.num_blocks, bs, free_order=w.free_order())
    ids = populate(lib, w)
    nblk = sum(-(-lib.length(s) // bs) for s in ids)
    block_bytes = 2 * Hkv * bs * D * w.elem_bytes  # K and V
    moved = nblk * block_bytes  # each way
    dk = torch.from_numpy(w.pool_values("k").view(np.int16)).view(torch.bfloat16).to(dev)
    dv = torch.from_numpy(w.pool_values("v").view(np.int16)).view(torch.bfloat16).to(dev)
    kst = torch.empty((nblk, Hkv, bs, D), dtype=torch.bfloat16, pin_memory=True)
    vst = torch.empty((nblk, Hkv, bs, D), dtype=torch.bfloat16, pin_memory=True)
    bl_out = torch.empty(nblk, dtype=torch.int32, pin_memory=True)
    bl_in = torch.empty(nblk, dtype=torch.int32, pin_memory=True)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def one_step(ev=None):
        pos = 0
        for s_ in ids:  # host: release every sequence's blocks, recording them in batch order
            b = lib.swap_out(s_)
            bl_out.numpy()[pos:pos + len(b)] = b
            pos += len(b)
        if ev:
            ev[0].record(stream)
        pa.pa_swap_out(dk, dv, bl_out, kst, vst, status=status, stream=stream)
        if ev:
            ev[1].record(stream)
        pos = 0
        for s_ in ids:  # host: fresh blocks for every sequence
            b = lib.swap_in(s_)
            bl_in.numpy()[pos:pos + len(b)] = b
            pos += len(b)
        if ev:
            ev[2].record(stream)
        pa.pa_swap_in(kst, vst, bl_in, dk, dv, status=status, stream=stream)
        if ev:
            ev[3].record(stream)
        stream.synchronize()  # the pinned block lists are rewritten by the next step

    for _ in range(Wm):
        one_step()
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4)) for _ in range(K)]
    clocks = ClockSampler(local_rank)
    clocks.start()
    for i in range(K):
        one_step(evs[i])
    clocks.stop()
    if status.item():
        raise SystemExit(f"device status word {int(status.item()):#x}")
    out_ms = [e[0].elapsed_time(e[1]) for e in evs]
    in_ms = [e[2].elapsed_time(e[3]) for e in evs]
    # the link's reference rate: copy-engine memcpy of the same bytes, device <-> pinned host
    dbuf = torch.empty(moved, dtype=torch.uint8, device=dev)
    hbuf = torch.empty(moved, dtype=torch.uint8, pin_memory=True)
    rates = {}
    for name, fn in (("d2h", lambda: hbuf.copy_(dbuf, non_blocking=True)),
                     ("h2d", lambda: dbuf.copy_(hbuf, non_blocking=True))):
        ts = []
        for _ in range(Wm + K):
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b_.record(stream)
            stream.synchronize()
            ts.append(a.elapsed_time(b_))
        rates[name] = moved / (statistics.median(ts[Wm:]) / 1e3) / 1e9
    total_s = reduce_max((sum(out_ms) + sum(in_ms)) / 1e3, dist, dev)
    value = reduce_sum(2.0 * moved * K, dist, dev) / total_s / 1e9
    out_gbs = moved / (statistics.median(out_ms) / 1e3) / 1e9
    in_gbs = moved / (statistics.median(in_ms) / 1e3) / 1e9
    peak = (rates["d2h"] + rates["h2d"]) / 2
    line = {
        "metric": SWAP_METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": total_s * 1e3 / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": f"synthetic, seeded: {WORKLOADS['gqa4_b64']}; every sequence swapped out and back",
        "config": {"workload": "swap_gqa4_b64_all", "blocks": nblk, "bytes_each_way": moved,
                   "swap_out_ms_median": statistics.median(out_ms), "swap_in_ms_median": statistics.median(in_ms),
                   "swap_out_gbs": out_gbs, "swap_in_gbs": in_gbs, "memcpy_d2h_gbs": rates["d2h"],
                   "memcpy_h2d_gbs": rates["h2d"],
                   "store": "pinned host memory, written and read by the kernels over the host link"},
        "roofline": {"bound": "host-link", "achieved": value, "peak": peak, "unit": "GB/s", "frac": value / peak,
                     "peak_source": "copy-engine memcpy between device and pinned host memory, same bytes, same run",
                     "kernel": "pa_swap_out + pa_swap_in (swap_blocks_kernel)", "traffic": None},
        "gpu_launches": 2 * K,
        "clocks": clocks.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# reference arm: the oracle on the host cores, same metric and workload
# ---------------------------------------------------------------------------
def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    from oracle.alloc_model import RefAllocator

    w = build_workload(args.workload, 0, 1, extra_steps=2)
    ref = RefAllocator(w.num_blocks, w.block_size, free_order=w.free_order().tolist())
    ids = populate(ref, w)
    B = len(ids)
    ref.append_batch(ids)
    lens = np.array([ref.length(s) for s in ids], np.int32)
    max_blocks = int(-(-int(lens.max()) // w.block_size))
    tables = np.zeros((B, max_blocks), np.int32)
    for i, s in enumerate(ids):
        t = ref.table(s)
        tables[i, : len(t)] = t
    k_pool, v_pool, q = w.pool_values("k"), w.pool_values("v"), w.queries(step=1)
    threads = os.cpu_count() or 1
    per_step = max(1, min(B, args.ref_seqs_per_step))
    times, tokens = [], []
    for i in range(args.warmup + args.steps):
        seqs = [(i * per_step + j) % B for j in range(per_step)]
        t0 = time.perf_counter()
        oracle.decode_attention(q, k_pool, v_pool, tables, lens, w.scale, seqs=seqs, threads=threads)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
            tokens.append(int(sum(int(lens[s]) for s in seqs)))
    value = sum(tokens) / sum(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": f"synthetic, seeded: {WORKLOADS[args.workload]}; blocks scattered by a seeded free-list order",
        "config": {"workload": w.name, "num_seqs_per_gpu": B, "num_q_heads": w.num_q_heads,
                   "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{per_step} of the {B} sequences per step (rotating), fp64 C oracle, "
                                   f"{threads} threads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_prefill_reference(args, rank, world):
    """The oracle's prefill of the same prompts on the host cores, each step a bounded sample of one prompt."""
    if rank != 0:
        return
    import synth

    w, P, L = prefill_setup(0, args.prompts)
    Hq, D = w.num_q_heads, w.head_dim
    from oracle.alloc_model import RefAllocator

    ref = RefAllocator(w.num_blocks, w.block_size, free_order=w.free_order().tolist())
    slots = []
    for p_ in range(P):
        ref.create(p_)
        slots.extend(ref.append(p_, L)[0])
    tables = np.zeros((P, -(-L // w.block_size)), np.int32)
    for p_ in range(P):
        t = ref.table(p_)
        tables[p_, : len(t)] = t
    lens = np.full(P, L, np.int32)
    q = synth.normal(synth.stream_seed(w.seed, 4242), P * L * Hq * D, "bf16").reshape(P * L, Hq, D)
    kn, vn = w.prompt_tokens("k")[: P * L], w.prompt_tokens("v")[: P * L]
    import oracle

    k_pool, v_pool = w.pool_values("k"), w.pool_values("v")
    oracle.reshape_and_cache(kn, vn, k_pool, v_pool, np.asarray(slots, np.int64))
    cu = np.arange(0, P * L + 1, L, dtype=np.int32)
    threads = os.cpu_count() or 1
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.prefill_attention(q, k_pool, v_pool, tables, lens, cu, w.scale, seqs=[i % P], threads=threads)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    value = L * len(times) / sum(times)
    line = {
        "impl": "reference", "metric": PREFILL_METRIC, "value": value, "unit": PREFILL_UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": f"synthetic, seeded: {P} prompts of {L} tokens, 32 query / 8 KV heads, d 128",
        "config": {"workload": f"prefill_p{P}_len{L}_hq{Hq}_hkv{w.num_kv_heads}_d{D}_bs{w.block_size}_bf16"},
        "cpu_baseline": {"value": value, "unit": PREFILL_UNIT, "cores": 1, "kind": "oracle",
                         "sample": "one whole prompt per step (rotating), fp64 C oracle, one thread"},
        "e2e": {"value": value, "unit": PREFILL_UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS),
                    help="headline workload (default: the largest single-GPU one); the others go to per_config")
    ap.add_argument("--no-per-config", action="store_true", help="measure the headline workload only")
    ap.add_argument("--per-config-steps", type=int, default=20)
    ap.add_argument("--per-config-cpu-seconds", type=float, default=2.0)
    ap.add_argument("--e2e-steps", type=int, default=128)
    ap.add_argument("--e2e-eager", action="store_true", help="e2e: launch the step's calls one by one, no CUDA graph")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-seqs-per-step", type=int, default=16)
    ap.add_argument("--path", choices=["decode", "prefill", "swap"], default="decode",
                    help="decode: the decode step (the headline); prefill: prompt prefill of the sampling prompts; "
                         "swap: the whole decode batch swapped to pinned host memory and back")
    ap.add_argument("--prompts", type=int, default=16, help="prefill path: prompts per step (at most 16)")
    ap.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                    help="decode path: pool element type (fp8: E4M3 codes with per-pool scales, bf16 queries)")
    ap.add_argument("--prefix-cached", action="store_true",
                    help="prefill path: the prompts share all but their last 7 tokens, already cached")
    ap.add_argument("--no-plan", action="store_true",
                    help="decode path: let the decode compute its work plan on the device instead of taking the "
                         "host-built one")
    ap.add_argument("--ctas-per-sm", type=int, default=0,
                    help="decode path: CTAs per SM of the decode grid (0: the per-path default); a comparison aid")
    ap.add_argument("--seg-units", type=int, default=0,
                    help="decode path: a segment's weight in the CTA range balance, a tile weighing 4 (0: the "
                         "per-path default); a comparison aid")
    ap.add_argument("--wave-skew", type=int, default=-1,
                    help="decode path: skew of the CTA shares by dispatch wave (-1: the per-path default, 0: "
                         "equal shares); a comparison aid")
    ap.add_argument("--merge-mode", type=int, choices=[0, 1, 2], default=0,
                    help="decode path: where split segments are merged (0: chosen per call, 1: in the decode "
                         "kernel, 2: by the merge kernel); a comparison aid")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("at least 3 warm-up steps")
    rank, world, local_rank = dist_env()
    if args.path == "swap":
        if args.impl == "reference":
            if rank == 0:
                print(json.dumps({"impl": "reference", "unavailable": "the swap path is plain block copies; the "
                                  "oracle has no arithmetic to time for it"}), flush=True)
        else:
            run_swap(args, rank, world, local_rank)
    elif args.path == "prefill":
        if args.impl == "reference":
            run_prefill_reference(args, rank, world)
        else:
            run_prefill(args, rank, world, local_rank)
    elif args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
