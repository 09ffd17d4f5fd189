#!/usr/bin/env python3
"""Benchmark of the FP8 E4M3 paged KV cache on GB300.

One step = one pass of the whole hot path over one batch: the fused
quantize-scatter of the step's new K/V rows (R per request) into the FP8 cache,
then paged GQA decode / verify attention over the cache (split-K partials, then
the combine).  Inputs are synthetic and seeded (workloads/), resident in HBM
before the timed region; L2 is flushed before every timed step (a 256 MiB write,
then a 256 MiB read that moves the write-back of those dirty lines out of the
timed step) and the step time is the sum of per-step CUDA-event intervals taken
on the launching stream.

Default workload: the decode batch -- 32 requests, context lengths uniform in
[1024, 8192], 32 query heads / 8 KV heads, head_dim 128, block size 16,
log-normal row magnitudes, one query row per request.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kvq|reference]
                  [--workload decode|verify|longctx|store|tiny|index|scores]

Prints one JSON line (rank 0).  --impl reference times the CPU oracle (oracle/)
on bounded samples of the same workload; it is a deliberately slow program, a
reported baseline and not the target.
"""
from __future__ import annotations

import argparse
import dataclasses
import ctypes
import hashlib
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

import workloads  # noqa: E402

METRIC = "paged FP8-KV decode attn: achieved HBM GB/s (% of 8 TB/s); KV rows quantized/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 256 << 20
STORE_LAYERS = 8          # layers of the prefill store stored in one timed step


class L2Flush:
    """Between timed steps: a write of a 256 MiB buffer (twice L2) evicts every
    line the previous step touched; a read of a second 256 MiB buffer then
    evicts the write's dirty lines, so their write-back happens here and not
    inside the next timed kernel, which starts with a clean L2 holding none of
    its data."""

    def __init__(self, dev):
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def __call__(self, i):
        self.w.fill_(i & 0xFF)
        torch.amax(self.r)

DESCRIPTIONS = {
    "tiny": "tiny: 1 request x 64 tokens, 32 q heads / 8 KV heads, head_dim 128, block 16",
    "decode": ("decode batch: 32 requests, context U[1024, 8192], 32 q heads / 8 KV heads, "
               "head_dim 128, block 16, log-normal rows, 1 query row per request"),
    "verify": ("MTP verify: 64 requests x 4 query rows, context 32768, 64 q heads / 8 KV heads, "
               "head_dim 128, block 64, 32 stacked rows per KV head"),
    "longctx": ("long-context split-K: 2 requests x 1,048,576 tokens, 32 q heads / 8 KV heads, "
                "head_dim 128, block 64"),
    "prefill": ("chunked prefill: 4 requests, each a 2,048-token chunk at the end of an "
                "8,192-token context (causal), 32 q heads / 8 KV heads, head_dim 128, block 64, "
                "log-normal rows"),
    "store": ("prefill store under CUDA graph: 16,384 tokens as strided K/V views of a fused "
              "qkv [16384, 6144], 1% outliers x50, zero rows, permuted int64 slot ids, block 64; "
              "one step stores 8 layers (8 qkv tensors into 8 caches, one launch each)"),
    "index": ("MXFP4 index-key store under CUDA graph: 262,144 rows of 128 bf16 values "
              "(N(0,1) x a log-normal magnitude per 32-dim group) into E2M1 codes (two a byte) + an E8M0 "
              "exponent per 32 dims, permuted int64 slot ids"),
    "scores": ("stacked index scores under CUDA graph: 64 requests x 4 query rows x 4 index "
               "heads (16 stacked vectors), context 32768, block 64, MXFP4 index keys, "
               "fp32 scores out"),
}

DEFAULT_STEPS = {"tiny": 2000, "decode": 5000, "verify": 1500, "longctx": 1500, "store": 5000,
                 "prefill": 300,
                 "index": 3000, "scores": 1500}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["kvq", "reference"], default="kvq")
    ap.add_argument("--workload", choices=list(DESCRIPTIONS), default="decode")
    ap.add_argument("--partition-tokens", type=int, default=0)
    ap.add_argument("--requests", type=int, default=0,
                    help="only the first N requests of the workload (a smaller case of the "
                         "same shape, for profiler captures); 0 = all")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--index-format", choices=["mxfp4", "fp8"], default="mxfp4",
                    help="index-key format of the scores workload")
    ap.add_argument("--no-per-config", action="store_true",
                    help="the default decode run only: skip timing the store, verify and "
                         "long-context configurations as well")
    ap.add_argument("--profile", action="store_true",
                    help="no L2 flush, clocks, e2e or CPU baseline: a short run for ncu")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# distributed (replicas: every rank runs its own copy of the workload)

def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, local, world


def dist_max(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# peaks, clocks, committed ncu traffic

def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0


def measured_tensor_peak():
    """Dense bf16 tensor TFLOP/s measured on this machine (sustained: the kernels
    run inside a long loop of steps), else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS_SUSTAINED, "fallback"


CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while it runs."""

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            self.sel = str(device_index)

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.sel, f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self, t_start: float, t_stop: float):
        if self.proc is None or not self.path:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[4:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for n, val in zip(names, r[2][1:]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows),
                "samples": len(rows), "reasons": sorted(reasons)}


def ncu_traffic(kernel: str, workload: str, source: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary (profiles/ncu_traffic.json), or None when the kernel's source file
    changed since the counters were taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            e = json.load(f)[f"{kernel}:{workload}"]
        with open(os.path.join(ROOT, source), "rb") as f:
            h = hashlib.sha256(f.read()).hexdigest()[:16]
        if e.get("source_sha256_16") != h:
            return None
        return float(e["bytes_per_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------------------
# workload on the device

class DeviceWorkload:
    def __init__(self, name: str, device, partition_tokens: int = 0, requests: int = 0):
        import fp8_paged_kv_kvq_gb300 as kvq
        self.kvq = kvq
        self.lib = kvq.load()
        self.name = name
        self.w = w = workloads.WORKLOADS[name]
        if 0 < requests < w.num_requests:
            self.w = w = dataclasses.replace(w, num_requests=requests)
        self.device = device
        self.stream = torch.cuda.Stream(device)
        H, D = w.num_kv_heads, w.head_dim
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        if name == "store":
            self._init_store()
            return
        self.lens = workloads.context_lengths(w)
        self.bt, nblk = workloads.block_tables(self.lens, w.block_size, w.seed)
        self.S = nblk * w.block_size
        self.cache = kvq.Cache.empty(self.S, H, D, w.block_size, device=device)
        ct = workloads.chunk_tokens(w)
        for r in range(w.num_requests):
            L = int(self.lens[r])
            slots_all = workloads.token_slots(self.bt, r, L, w.block_size)
            for c0 in range(0, L, ct):
                n = min(ct, L - c0)
                k, v = workloads.request_kv(w, r, c0, n, device=device)
                kvq.quantize_scatter(self.cache, k, v,
                                     torch.from_numpy(slots_all[c0:c0 + n]).to(device), self.err)
        R = w.rows_per_request
        # the step's new rows: the last R tokens of every request (already in
        # the cache with the same values, so storing them again is idempotent)
        ks, vs, sl = [], [], []
        for r in range(w.num_requests):
            L = int(self.lens[r])
            k, v = workloads.request_kv(w, r, L - R, R, device=device)
            ks.append(k)
            vs.append(v)
            sl.append(workloads.token_slots(self.bt, r, L, w.block_size)[L - R:])
        self.new_k = torch.cat(ks).contiguous()
        self.new_v = torch.cat(vs).contiguous()
        self.new_slots = torch.from_numpy(np.concatenate(sl)).to(device)
        self.q = workloads.queries(w, device=device)
        self.bt_d = torch.from_numpy(self.bt).to(device)
        self.cl_d = torch.from_numpy(self.lens).to(device)
        self.max_ctx = int(self.lens.max())
        # partition size passed to the library: 0 leaves it (and the kernel) to
        # the library; self.P is the partition it would use for partitioned kernels
        self.P_arg = partition_tokens
        self.P = partition_tokens or kvq.paged_decode_partition_tokens(
            w.num_requests, R, w.num_q_heads, H, w.block_size, self.max_ctx)
        self.n_parts = (self.max_ctx + self.P - 1) // self.P
        self.balanced = self.P_arg == 0 and self._balanced_mode()
        # the load-balanced kernel stores the step's new rows itself
        # (kvq_paged_decode_append_partials): the step has no store launch
        self.fused = self.balanced
        # more than 8 stacked rows per KV head, partition left to the library:
        # the rows-on-M tensor-core kernel, which merges its pieces itself
        rows = R * w.group
        self.rows_kernel = (self.P_arg == 0 and rows > 8 and rows <= 8192
                            and w.block_size >= 16 and H % 4 == 0 and w.num_requests <= 1024)
        need = kvq.paged_decode_workspace_size(w.num_requests, R, w.num_q_heads, H, D,
                                               w.block_size, self.max_ctx, self.P_arg)
        self.ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=device)
        self.out = torch.empty_like(self.q)
        torch.cuda.synchronize(device)
        assert int(self.err.item()) == 0, "setup store reported an error"
        self._bind()

    def _init_store(self):
        """STORE_LAYERS layers of a prefill: each layer its own fused qkv
        tensor (the workload's recipe, the same values) and its own cache, all
        stored in one step, one launch per layer."""
        w = self.w
        qkv, _, _, slots, S = workloads.store_qkv(w, device=self.device)
        Hq, H, D = w.num_q_heads, w.num_kv_heads, w.head_dim
        self.layers = STORE_LAYERS
        self.qkvs = [qkv] + [qkv.clone() for _ in range(self.layers - 1)]
        self.qkv = qkv
        self.new_ks = [x[:, Hq * D:(Hq + H) * D].view(-1, H, D) for x in self.qkvs]
        self.new_vs = [x[:, (Hq + H) * D:].view(-1, H, D) for x in self.qkvs]
        self.new_k, self.new_v = self.new_ks[0], self.new_vs[0]
        self.new_slots = slots
        self.S = S
        self.n_parts = 0
        self.caches = [self.kvq.Cache.empty(S, H, D, w.block_size, device=self.device)
                       for _ in range(self.layers)]
        self.cache = self.caches[0]
        torch.cuda.synchronize(self.device)
        self._bind()

    def _bind(self):
        """Pre-built ctypes argument lists for the C-ABI calls of one step."""
        w, P = self.w, ctypes.c_void_p
        sp = P(self.stream.cuda_stream)
        if self.name == "store":
            self._csts = [c.struct() for c in self.caches]
            T = self.new_k.shape[0]
            self._q_args_layers = [
                (ctypes.byref(cst), P(k.data_ptr()), k.stride(0), P(v.data_ptr()), v.stride(0),
                 T, P(self.new_slots.data_ptr()), P(self.err.data_ptr()), sp)
                for cst, k, v in zip(self._csts, self.new_ks, self.new_vs)]
            return
        self._cst = self.cache.struct()
        T = self.new_k.shape[0]
        self._q_args = (ctypes.byref(self._cst), P(self.new_k.data_ptr()), self.new_k.stride(0),
                        P(self.new_v.data_ptr()), self.new_v.stride(0), T,
                        P(self.new_slots.data_ptr()), P(self.err.data_ptr()), sp)
        R, N = w.rows_per_request, w.num_requests
        self._p_args = (ctypes.byref(self._cst), P(self.q.data_ptr()), N, R, w.num_q_heads,
                        P(self.bt_d.data_ptr()), self.bt.shape[1], P(self.cl_d.data_ptr()),
                        self.max_ctx, ctypes.c_float(w.sm_scale), self.P_arg, P(self.out.data_ptr()),
                        P(self.ws.data_ptr()), self.ws.numel(), P(self.err.data_ptr()), sp)
        self._a_args = (ctypes.byref(self._cst), P(self.new_k.data_ptr()), self.new_k.stride(0),
                        P(self.new_v.data_ptr()), self.new_v.stride(0)) + self._p_args[1:]
        self._c_args = (ctypes.byref(self._cst), N, R, w.num_q_heads, self.bt.shape[1],
                        P(self.cl_d.data_ptr()), self.max_ctx, self.P_arg, P(self.out.data_ptr()),
                        P(self.ws.data_ptr()), self.ws.numel(), sp)

    def _balanced_mode(self):
        """Whether the library runs the load-balanced kernel for this shape when
        left to choose: at most 8 stacked rows, pages of >= 16 tokens, KV heads
        in groups of 4, at most 1024 requests, a CTA's chunks within its 520
        block ids, and a page-major partition grid under 9 CTAs per SM."""
        w = self.w
        rows = w.rows_per_request * w.group
        sms = torch.cuda.get_device_properties(self.device).multi_processor_count
        cmax = (self.max_ctx + 15) // 16
        hg = w.num_kv_heads // 4
        total_ub = w.num_requests * hg * (cmax + 5)
        per_cta = (total_ub + 3 * sms - 1) // (3 * sms)
        per_cta_w = (total_ub * 135 + 384 * sms - 1) // (384 * sms) + 1   # weighted ranges
        b = max(per_cta, (cmax + 14) // 15, per_cta_w)
        page_ctas = hg * self.n_parts * w.num_requests
        return (rows <= 8 and w.block_size >= 16 and w.num_kv_heads % 4 == 0
                and 1 <= w.num_requests <= 1024 and b * 16 // w.block_size + 2 <= 520
                and total_ub < 2 ** 31 and page_ctas < 9 * sms)

    def partials_kernel(self):
        """(kernel, source) the library launches for this shape's partials:
        the load-balanced kernel when the library picks it (see _stream_mode);
        for at most 8 stacked rows per KV head the page-major kernel when its
        grid (4 heads per CTA) is at least 9 CTAs per SM, else the skinny one
        (pages of at least 8 tokens); with an explicit partition the tcgen05
        kernel for 9..32 rows (pages
        of 16..128 tokens, KV heads a multiple of 4, partitions a multiple of
        128 tokens); else the general one."""
        w = self.w
        if self.balanced:
            return "attn_stream_kernel", "fp8_paged_kv_kvq_gb300/csrc/kvq_attention_stream.cu"
        rows = w.rows_per_request * w.group
        if self.rows_kernel:
            return "attn_rows_kernel", "fp8_paged_kv_kvq_gb300/csrc/kvq_attention_rows.cu"
        page_ctas = (w.num_kv_heads // 4) * self.n_parts * w.num_requests
        sms = torch.cuda.get_device_properties(self.device).multi_processor_count
        if (rows <= 8 and w.block_size >= 16 and w.num_kv_heads % 4 == 0
                and page_ctas >= 9 * sms):
            return "attn_page_kernel", "fp8_paged_kv_kvq_gb300/csrc/kvq_attention_page.cu"
        if rows <= 8 and w.block_size >= 8:
            return "attn_skinny_kernel", "fp8_paged_kv_kvq_gb300/csrc/kvq_attention_skinny.cu"
        if (rows <= 32 and 16 <= w.block_size <= 128 and w.num_kv_heads % 4 == 0
                and self.P % 128 == 0):
            return "attn_tc_kernel", "fp8_paged_kv_kvq_gb300/csrc/kvq_attention_tc.cu"
        return "attn_partials_kernel", "fp8_paged_kv_kvq_gb300/csrc/kvq_attention.cu"

    # the launches of a step, through the C ABI
    def quantize(self):
        for args in (self._q_args_layers if self.name == "store" else (self._q_args,)):
            st = self.lib.kvq_quantize_scatter(*args)
            if st:
                raise RuntimeError(f"kvq_quantize_scatter: status {st}")

    def partials(self):
        st = self.lib.kvq_paged_decode_partials(*self._p_args)
        if st:
            raise RuntimeError(f"kvq_paged_decode_partials: status {st}")

    def append_partials(self):
        st = self.lib.kvq_paged_decode_append_partials(*self._a_args)
        if st:
            raise RuntimeError(f"kvq_paged_decode_append_partials: status {st}")

    def store_and_partials(self, between=None):
        """The step's store of its new rows and the attention's split-K launch:
        one launch where the load-balanced kernel stores the rows itself, else
        the store's launch, then (after `between`, an event record) the
        partials."""
        if self.fused:
            if between is not None:
                between()
            self.append_partials()
            return
        self.quantize()
        if between is not None:
            between()
        self.partials()

    def combine(self):
        st = self.lib.kvq_paged_decode_combine(*self._c_args)
        if st:
            raise RuntimeError(f"kvq_paged_decode_combine: status {st}")

    @property
    def store_launches(self):
        return self.layers if self.name == "store" else 1

    @property
    def launches_per_step(self):
        if self.name == "store":
            return self.layers
        if self.rows_kernel:
            return 2
        return (1 if self.fused else 2) + (1 if self.n_parts > 1 else 0)

    # algorithmic bytes: attention = codes + scales + q + out + block tables +
    # context lengths; store = bf16 K/V read + codes + scales + slot ids, per
    # layer
    def store_bytes_per_launch(self):
        w = self.w
        T = self.new_k.shape[0]
        H, D = w.num_kv_heads, w.head_dim
        # slot ids: none when the attention launch stores the rows at their
        # block-table positions
        return T * H * (2 * D * 2 + 2 * D + 2 * 4) + (0 if getattr(self, "fused", False) else T * 8)

    def store_bytes(self):
        return self.store_launches * self.store_bytes_per_launch()

    def attn_bytes(self):
        if self.name == "store":
            return 0
        w = self.w
        H, D = w.num_kv_heads, w.head_dim
        tok = int(self.lens.sum())
        bt = sum((int(L) + w.block_size - 1) // w.block_size for L in self.lens) * 4
        return tok * H * 2 * (D + 4) + 2 * self.q.numel() * 2 + bt + 4 * w.num_requests

    def attn_flops(self):
        """Useful flops of the attention: 2 D for q.k and 2 D for p v per
        (query row, query head, token it sees)."""
        if self.name == "store":
            return 0
        w = self.w
        R, D = w.rows_per_request, w.head_dim
        seen = sum(sum(max(0, min(int(L), int(L) - R + 1 + i)) for i in range(R))
                   for L in self.lens)
        return seen * w.num_q_heads * 4 * D

    def rows_quantized(self):
        return self.store_launches * self.new_k.shape[0] * self.w.num_kv_heads * 2

    def tokens(self):
        return self.store_launches * self.new_k.shape[0]


# ---------------------------------------------------------------------------
# the GPU arm

# the other configurations the default (decode) run also times, with their steps
PER_CONFIG_STEPS = {"store": 600, "verify": 200, "longctx": 300, "prefill": 100}


def run_kvq(args, rank, local, world):
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    K = args.steps if args.steps is not None else DEFAULT_STEPS[args.workload]
    W = max(3, args.warmup if args.warmup is not None else min(50, max(3, K // 10)))
    wl = DeviceWorkload(args.workload, dev, args.partition_tokens, args.requests)
    with torch.cuda.stream(wl.stream):
        res = _run_kvq_on_stream(args, rank, local, world, dev, wl, K, W)
    del wl
    torch.cuda.empty_cache()
    if (args.workload == "decode" and not args.profile and not args.no_per_config
            and args.requests <= 0 and args.partition_tokens == 0):
        # the store, verify and long-context configurations, each timed the same
        # way (its own clocks, roofline and per-kernel times); the headline
        # value stays the decode batch's
        res["per_config"] = {}
        for name, k in PER_CONFIG_STEPS.items():
            sub = argparse.Namespace(**vars(args))
            sub.workload, sub.steps, sub.warmup = name, k, 3
            sub.no_e2e = sub.no_cpu_baseline = True
            sub.no_per_config = True
            r = run_kvq(sub, rank, local, world)
            keep = ("value", "unit", "ms_per_step", "pct_of_8tbs", "pct_of_hbm_peak",
                    "kv_rows_quantized_per_s", "tokens_per_s", "kernels_us", "roofline",
                    "clocks", "steps", "warmup")
            entry = {k2: r[k2] for k2 in keep if k2 in r}
            entry["workload"] = r["config"]["workload"]
            for k2 in ("partition_tokens", "partitions", "split", "layers"):
                if k2 in r["config"]:
                    entry[k2] = r["config"][k2]
            res["per_config"][name] = entry
        st = res["per_config"]["store"]
        res["decode_step_rows_quantized_per_s"] = res["kv_rows_quantized_per_s"]
        res["kv_rows_quantized_per_s"] = st["kv_rows_quantized_per_s"]
        res["kv_rows_quantized_note"] = (
            "KV rows quantized/s of the prefill store configuration (16,384 tokens x 8 KV "
            "heads x K and V per layer, 8 layers per CUDA-graph step); the decode step's own "
            "new rows are in decode_step_rows_quantized_per_s")
    return res


def _run_kvq_on_stream(args, rank, local, world, dev, wl, K, W):
    stream = wl.stream
    flush = None if args.profile else L2Flush(dev)
    graph = None
    if args.workload == "store":
        wl.quantize()
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            wl.quantize()
        torch.cuda.synchronize(dev)

    def step(evs=None, split=False):
        # split: events between the launches too (per-kernel durations); they
        # are stream operations that keep a launch from starting while the
        # previous kernel drains, so the step timing records only its ends
        if evs is not None:
            evs[0].record(stream)
        if graph is not None:
            graph.replay()
            if evs is not None:
                for e in evs[1:]:
                    e.record(stream)
            return
        wl.store_and_partials((lambda: evs[1].record(stream)) if split else None)
        if split:
            evs[2].record(stream)
        wl.combine()
        if evs is not None:
            evs[3].record(stream)

    for i in range(W):
        if flush is not None:
            flush(i & 0xFF)
        step()
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    peak, peak_src = measured_peaks()
    sampler = ClockSampler(local) if not args.profile else None
    dist_barrier(world)
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.start()
    wall0 = time.perf_counter()
    torch.cuda.nvtx.range_push("kvq_timed")      # lets a profiler select the timed launches
    for i in range(K):
        if flush is not None:
            flush((i + 7) & 0xFF)
        step(evs[i])
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize(dev)
    wall1 = time.perf_counter()
    if sampler:
        sampler.stop()
    dist_barrier(world)
    st = [e[0].elapsed_time(e[3]) for e in evs]
    step_ms = dist_max(sum(st) / K, world)
    # per-kernel durations: a second pass of K steps, events between the launches
    kevs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    for i in range(K):
        if flush is not None:
            flush((i + 11) & 0xFF)
        step(kevs[i], split=True)
    torch.cuda.synchronize(dev)
    st_q = [e[0].elapsed_time(e[1]) for e in kevs]
    st_p = [e[1].elapsed_time(e[2]) for e in kevs]
    st_c = [e[2].elapsed_time(e[3]) for e in kevs]
    if int(wl.err.item()) != 0:
        raise RuntimeError("device error flags set during the benchmark")

    step_bytes = wl.store_bytes() + wl.attn_bytes()
    value = world * step_bytes / (step_ms * 1e-3) / 1e9
    res = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": DESCRIPTIONS[args.workload],
            "name": args.workload,
            "l2": ("flushed before every timed step (256 MiB write, then a 256 MiB read "
                   "that takes the write-back of its dirty lines out of the step); step "
                   "time = sum of "
                   "per-step CUDA-event intervals (events at the step's ends only; "
                   "per-kernel times from a second pass of K steps with events between "
                   "the launches)") if flush is not None else
                  "not flushed (profile mode)",
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
            "storage": "e4m3 codes (uint8) + fp32 row scales; bf16 q/out; QK^T on e4m3 tensor "
                       "cores (q as two exact e4m3 pieces), PV on f16 tensor cores, fp32 "
                       "accumulate",
        },
        "pct_of_8tbs": round(100.0 * value / world / NOMINAL_HBM_GBS, 2),
        "pct_of_hbm_peak": round(100.0 * value / world / peak, 2),
        "kv_rows_quantized_per_s": round(world * wl.rows_quantized() / (step_ms * 1e-3), 1),
        "tokens_per_s": round(world * wl.tokens() / (step_ms * 1e-3), 1),
        "kernels_us": {"quantize_scatter": round(1e3 * sum(st_q) / K, 3)},
        "gpu_launches": K * wl.launches_per_step,   # in the step-timed pass
        "wall_s_timed_region": round(wall1 - wall0, 3),
    }
    if args.workload != "store":
        if wl.balanced:
            res["config"]["split"] = ("load-balanced: the batch's 16-token chunks split over a "
                                      "persistent grid (3 CTAs per SM, ranges weighted by the "
                                      "grid's dispatch thirds)")
        elif wl.rows_kernel:
            res["config"]["split"] = ("load-balanced: the batch's 128-token chunks split evenly "
                                      "over a persistent grid (1 CTA per SM), cut units merged "
                                      "in the same launch")
        else:
            res["config"]["partition_tokens"] = wl.P
            res["config"]["partitions"] = wl.n_parts
        res["kernels_us"]["paged_decode_partials"] = round(1e3 * sum(st_p) / K, 3)
        res["kernels_us"]["paged_decode_combine"] = round(1e3 * sum(st_c) / K, 3)
        dom_ms, dom_bytes = sum(st_p) / K, wl.attn_bytes()
        if wl.fused:
            res["config"]["store"] = ("fused: the load-balanced kernel stores the step's new "
                                      "rows itself (kvq_paged_decode_append_partials)")
            res["kernels_us"]["quantize_scatter_note"] = (
                "no store launch: paged_decode_partials is the append launch that stores "
                "the new rows and runs the split-K attention")
            dom_bytes += wl.store_bytes_per_launch()
        dom_name, dom_src = wl.partials_kernel()
    else:
        # one graph replay stores every layer: a launch's time is the step's share
        dom_ms, dom_bytes = sum(st_q) / K / wl.layers, wl.store_bytes_per_launch()
        dom_name, dom_src = "quantize_scatter_kernel", "fp8_paged_kv_kvq_gb300/csrc/kvq_quantize.cu"
        res["config"]["layers"] = wl.layers
        res["kernels_us"]["quantize_scatter"] = round(1e3 * dom_ms, 3)
        res["kernels_us"]["quantize_scatter_note"] = (
            f"per launch: the {wl.layers}-launch graph replay divided by {wl.layers}")
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    if args.workload == "prefill":
        # compute-bound: many rows share each KV byte.  q.k runs as two e4m3
        # pieces at twice the bf16 rate, p v on f16 at the bf16 rate, so the
        # useful flops at the bf16 peak take the time of the executed ones
        tpeak, tsrc = measured_tensor_peak()
        flops = wl.attn_flops()
        tf = flops / (dom_ms * 1e-3) / 1e12
        res["attn_tflops"] = round(tf, 2)
        res["roofline"] = {
            "kernel": dom_name, "bound": "tensor", "achieved": round(tf, 2), "peak": tpeak,
            "peak_source": ("measured (MEASURED_PEAKS.json bf16_tflops_sustained; the q.k "
                            "pieces on e4m3 at twice the bf16 rate and p.v on f16 make the "
                            "useful flops' peak the bf16 one)" if tsrc == "measured"
                            else "fallback 1.7 PFLOP/s"),
            "unit": "TFLOP/s", "frac": round(tf / tpeak, 4),
            "algorithmic_flops_per_launch": flops,
            "hbm_gbs_of_algorithmic_bytes": round(achieved, 2),
            "traffic": ncu_traffic(dom_name, args.workload, dom_src),
        }
    else:
        res["roofline"] = {
            "kernel": dom_name,
            "bound": "hbm",
            "achieved": round(achieved, 2),
            "peak": peak,
            "peak_source": ("measured (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                            else "fallback 6.8 TB/s"),
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "algorithmic_bytes_per_launch": dom_bytes,
            "traffic": ncu_traffic(dom_name, args.workload, dom_src),
        }
    if sampler:
        res["clocks"] = sampler.summary(wall0, wall1)
    if not args.profile and not args.no_e2e:
        n_e2e = max(20, min(K, 300))
        res["e2e"] = (run_e2e_store(wl, dev, n_e2e, world) if args.workload == "store"
                      else run_e2e(wl, dev, n_e2e, world))
    if rank == 0 and world == 1 and not args.profile and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(args.workload, budget_s=12.0)
    return res


def _timed(stream, dev, K, body, flush):
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    for i in range(K):
        if flush is not None:
            flush(i & 0xFF)
        ev[i][0].record(stream)
        body()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    return sum(a.elapsed_time(b) for a, b in ev) / K


def run_e2e(wl: DeviceWorkload, dev, K, world):
    """The same step through the C ABI with host buffers: the step's inputs
    (q, new K/V rows, slot ids where the store takes them, block tables,
    context lengths) are packed in one pinned host buffer and copied to the
    device in one transfer, the output read back, inside the timed region.
    The workload's input tensors are rebound as views into the device buffer."""
    names = ("q", "new_k", "new_v", "bt_d", "cl_d") if wl.fused else \
        ("q", "new_k", "new_v", "new_slots", "bt_d", "cl_d")
    layout, total = [], 0
    for name in names:
        t = getattr(wl, name).contiguous()
        nb = t.numel() * t.element_size()
        layout.append((name, total, nb, t))
        total = (total + nb + 255) // 256 * 256
    dev_buf = torch.empty(total, dtype=torch.uint8, device=dev)
    host_buf = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    for name, off, nb, t in layout:
        host_buf[off:off + nb].copy_(t.reshape(-1).view(torch.uint8).cpu())
        setattr(wl, name, dev_buf[off:off + nb].view(t.dtype).view(t.shape))
    wl._bind()
    out_h = torch.empty(wl.out.shape, dtype=wl.out.dtype, pin_memory=True)
    h2d = sum(nb for _, _, nb, _ in layout)
    d2h = out_h.numel() * out_h.element_size()
    flush = L2Flush(dev)

    def body():
        dev_buf.copy_(host_buf, non_blocking=True)
        wl.store_and_partials()
        wl.combine()
        out_h.copy_(wl.out, non_blocking=True)

    for _ in range(3):
        body()
    torch.cuda.synchronize(dev)
    ms = dist_max(_timed(wl.stream, dev, K, body, flush), world)
    value = world * (wl.store_bytes() + wl.attn_bytes()) / (ms * 1e-3) / 1e9
    return {"value": round(value, 2), "unit": "GB/s", "ms_per_step": round(ms, 5),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "h2d_copies_per_step": 1}


def run_e2e_store(wl: DeviceWorkload, dev, K, world):
    """Every layer's K/V part of the qkv and the slot ids copied in from pinned
    host memory, the layers stored, the last layer's K scale plane read back."""
    w = wl.w
    Hq, D = w.num_q_heads, w.head_dim
    host_kv = [torch.empty(x[:, Hq * D:].shape, dtype=x.dtype, pin_memory=True).copy_(
        x[:, Hq * D:]) for x in wl.qkvs]
    host_slots = torch.empty(wl.new_slots.shape, dtype=torch.int64,
                             pin_memory=True).copy_(wl.new_slots)
    out_h = torch.empty(wl.cache.k_scales.shape, dtype=torch.float32, pin_memory=True)
    h2d = sum(h.numel() * 2 for h in host_kv) + host_slots.numel() * 8
    d2h = out_h.numel() * 4
    flush = L2Flush(dev)

    def body():
        for x, h in zip(wl.qkvs, host_kv):
            x[:, Hq * D:].copy_(h, non_blocking=True)
        wl.new_slots.copy_(host_slots, non_blocking=True)
        wl.quantize()
        out_h.copy_(wl.caches[-1].k_scales, non_blocking=True)

    for _ in range(3):
        body()
    torch.cuda.synchronize(dev)
    ms = dist_max(_timed(wl.stream, dev, K, body, flush), world)
    value = world * wl.store_bytes() / (ms * 1e-3) / 1e9
    return {"value": round(value, 2), "unit": "GB/s", "ms_per_step": round(ms, 5),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


# ---------------------------------------------------------------------------
# the CPU oracle on bounded samples (cpu_baseline and the reference arm)

class OracleSampler:
    """Units of the workload the oracle processes one at a time: a unit is one
    (request, query row, query head) attention output plus the quantize-scatter
    of that request's new rows for the head's KV head.  The oracle's cache of a
    request is built from the same seeded bf16 recipe, untimed, the first time a
    unit needs it."""

    def __init__(self, name: str, token_cap: int | None = None):
        import oracle
        self.oracle = oracle
        self.w = w = workloads.WORKLOADS[name]
        self.name = name
        self.token_cap = token_cap
        if name == "store":
            return
        self.lens = workloads.context_lengths(w)
        self.bt, nblk = workloads.block_tables(self.lens, w.block_size, w.seed)
        self.S = nblk * w.block_size
        self.q = workloads.bf16_bits(workloads.queries(w, device="cpu"))
        self._key = None
        # request-major order: consecutive units share one oracle cache
        self.units = [(r, i, h * w.group + g) for r in range(w.num_requests)
                      for h in range(w.num_kv_heads) for g in range(w.group)
                      for i in range(w.rows_per_request)]
        self.pos = 0

    def _request_cache(self, r):
        """The oracle's cache of request r, all KV heads, its L tokens at slots
        0..L-1 (an identity block table), built untimed on first use."""
        if self._key != r:
            w = self.w
            L, D, H = int(self.lens[r]), w.head_dim, w.num_kv_heads
            nb = (L + w.block_size - 1) // w.block_size
            self._oc = None
            oc = self.oracle.empty_cache(nb * w.block_size, H, D)
            dev = "cuda" if torch.cuda.is_available() else "cpu"
            k, v = workloads.request_kv(w, r, 0, L, device=dev)
            kb, vb = workloads.bf16_bits(k).reshape(-1), workloads.bf16_bits(v).reshape(-1)
            self.oracle.quantize_scatter(kb, H * D, vb, H * D, L, H, D,
                                         np.arange(L, dtype=np.int64), oc)
            R = w.rows_per_request
            self._new = (kb[(L - R) * H * D:].reshape(R, H, D),
                         vb[(L - R) * H * D:].reshape(R, H, D))
            self._bt = np.arange(nb, dtype=np.int32)[None, :]
            self._oc = oc
            self._key = r
        return self._oc

    def next_unit(self):
        """Prepare the next unit (untimed); returns (callable, algorithmic bytes
        of the unit: its even share of its request's step bytes)."""
        w = self.w
        r, i, hq = self.units[self.pos % len(self.units)]
        self.pos += 1
        h = hq // w.group
        oc = self._request_cache(r)
        L = int(self.lens[r])
        Lc = L if self.token_cap is None else min(L, self.token_cap)
        R, D, Hq = w.rows_per_request, w.head_dim, w.num_q_heads
        lens = np.array([Lc], dtype=np.int32)
        qreq = self.q[r * R:(r + 1) * R]
        bt = self._bt
        kb = np.ascontiguousarray(self._new[0][:, h]).reshape(-1)
        vb = np.ascontiguousarray(self._new[1][:, h]).reshape(-1)
        scratch = self.oracle.empty_cache(R, 1, D)
        new_slots = np.arange(R, dtype=np.int64)
        ora = self.oracle
        unit = np.array([[0, i, hq]], dtype=np.int32)

        def run():
            ora.quantize_scatter(kb, D, vb, D, R, 1, D, new_slots, scratch)
            ora.paged_attention_units(oc, qreq, 1, R, Hq, bt, lens, w.block_size, w.sm_scale,
                                      unit)

        H, Hq = w.num_kv_heads, w.num_q_heads
        req = (Lc * H * 2 * (D + 4) + ((Lc + w.block_size - 1) // w.block_size) * 4 + 4
               + R * Hq * 2 * D * 2 + R * H * (2 * D * 2 + 2 * D + 2 * 4) + R * 8)
        return run, req / (R * Hq)

    def store_run(self, rows: int, part: int = 0):
        """Store workload: quantise about `rows` (token, head) rows of the qkv,
        tokens [part T, (part + 1) T) (wrapping), so concurrent runs with
        different `part` write disjoint slots."""
        w = self.w
        if not hasattr(self, "_qkv"):
            qkv, _, _, slots, _ = workloads.store_qkv(w, device="cpu")
            self._qkv = workloads.bf16_bits(qkv)
            self._slots = slots.numpy()
            self._cache = self.oracle.empty_cache(self._qkv.shape[0], w.num_kv_heads,
                                                  w.head_dim)
        Hq, H, D = w.num_q_heads, w.num_kv_heads, w.head_dim
        n_tok = self._qkv.shape[0]
        T = min(max(1, rows // (2 * H)), n_tok)
        t0 = (part * T) % max(1, n_tok - T + 1)
        pitch = self._qkv.shape[1]
        flat = self._qkv[t0:].reshape(-1)
        slots = self._slots[t0:t0 + T]
        ora, cache = self.oracle, self._cache

        def run():
            ora.quantize_scatter(flat[Hq * D:], pitch, flat[(Hq + H) * D:], pitch, T, H, D,
                                 slots, cache)

        return run, T * H * (2 * D * 2 + 2 * D + 8) + T * 8


def host_cores() -> int:
    """Host threads this process may run on (its CPU affinity)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def run_parallel(runs, cores: int) -> float:
    """Wall-clock seconds to run the prepared callables on `cores` host threads
    (the oracle's C calls release the GIL, so they run concurrently)."""
    import concurrent.futures
    t0 = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(max_workers=cores) as ex:
        for f in [ex.submit(r) for r in runs]:
            f.result()
    return time.perf_counter() - t0


def cpu_baseline(name: str, budget_s: float):
    """The oracle, as it stands, over a bounded sample of the workload: on one
    host thread, then on every host core (one unit per thread at a time)."""
    s = OracleSampler(name)
    cores = host_cores()
    unit_rows = 2 * 8 * 512

    def one(part=0):
        return s.store_run(unit_rows, part) if name == "store" else s.next_unit()

    # one thread
    done_bytes, elapsed, units = 0.0, 0.0, 0
    setup0 = time.perf_counter()
    while elapsed < budget_s / 2 and time.perf_counter() - setup0 < 2 * budget_s:
        run, nb = one()
        t0 = time.perf_counter()
        run()
        elapsed += time.perf_counter() - t0
        done_bytes += nb
        units += 1
    single = done_bytes / elapsed / 1e9
    # every core: batches of `cores` units prepared untimed, then run at once
    s.pos = 0
    p_bytes, p_wall, p_units, batch = 0.0, 0.0, 0, 0
    setup0 = time.perf_counter()
    while p_wall < budget_s / 2 and time.perf_counter() - setup0 < 2 * budget_s:
        prepared = [one(batch * cores + i) for i in range(cores)]
        p_wall += run_parallel([r for r, _ in prepared], cores)
        p_bytes += sum(nb for _, nb in prepared)
        p_units += len(prepared)
        batch += 1
    what = ("(request, query row, query head) units: attention output over the full context "
            "plus the unit's share of the new-row store" if name != "store"
            else "blocks of 512 tokens (8192 rows) of the store")
    return {"value": round(p_bytes / p_wall / 1e9, 5), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{p_units} {what}, {cores} at a time on {cores} host threads "
                      f"({p_wall:.1f} s wall, {p_bytes / 1e6:.1f} MB algorithmic); one "
                      f"thread: {units} units in {elapsed:.1f} s",
            "single_thread": {"value": round(single, 5), "unit": "GB/s", "cores": 1}}


def run_reference(args, rank, world):
    """--impl reference: the oracle on the host, each step a bounded sample
    run on every host core (one unit per thread)."""
    if rank != 0:
        return None
    K = args.steps if args.steps is not None else 60
    W = max(3, args.warmup if args.warmup is not None else 3)
    name = args.workload
    cores = host_cores()
    per_step_s = min(2.0, 150.0 / (K + W))   # W + K steps within a few minutes
    s = OracleSampler(name)
    if name != "store":
        s.token_cap = 1024                     # calibrate cost per cached token
        run, _ = s.next_unit()
        t0 = time.perf_counter()
        run()
        per_tok = (time.perf_counter() - t0) / 1024
        s.token_cap = max(16, int(per_step_s / max(per_tok, 1e-9)))
        s.pos = 0
    rows_per_step = 16 * 8 * 2
    part = [0]

    def one():
        part[0] += 1
        return s.store_run(rows_per_step, part[0]) if name == "store" else s.next_unit()

    for _ in range(W):
        run_parallel([one()[0] for _ in range(cores)], cores)
    total_t, total_b = 0.0, 0.0
    for _ in range(K):
        prepared = [one() for _ in range(cores)]
        total_t += run_parallel([r for r, _ in prepared], cores)
        total_b += sum(nb for _, nb in prepared)
    value = total_b / total_t / 1e9
    if name == "store":
        sample = f"each step {cores} x {rows_per_step} rows of the store, one block per thread"
    else:
        max_len = int(s.lens.max())
        ctx = ("its full context" if s.token_cap >= max_len
               else f"its context capped at {s.token_cap} tokens")
        sample = (f"each step {cores} (request, query row, query head) units, one per host "
                  f"thread, each over {ctx}, plus its share of the new-row store")
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 5), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(1e3 * total_t / K, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": DESCRIPTIONS[name], "name": name},
        "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


# ---------------------------------------------------------------------------
# the index-key store (MXFP4)

INDEX_TOKENS = 262144
INDEX_ROW_BYTES = 128 * 2 + 64 + 4 + 8      # bf16 row read, codes, exponents, slot id
INDEX_METRIC = "MXFP4 index-key store: achieved HBM GB/s (% of 8 TB/s); rows quantized/s"


def index_inputs():
    """Seeded bf16 rows [262144, 128] (N(0,1) times exp(2 N(0,1)) per 32-dim
    group) and a permutation of the slots, on the host."""
    g = torch.Generator().manual_seed(5)
    x = torch.randn(INDEX_TOKENS, 4, 32, generator=g) * torch.exp(
        2.0 * torch.randn(INDEX_TOKENS, 4, 1, generator=g))
    slots = torch.randperm(INDEX_TOKENS, generator=g).to(torch.int64)
    return x.reshape(INDEX_TOKENS, 128).to(torch.bfloat16), slots


def index_oracle_rate(budget_s: float, x=None, cores: int = 1):
    """The oracle's MXFP4 quantisation over a bounded sample of the rows, in
    4096-row chunks, `cores` chunks at a time on as many host threads:
    (GB/s of algorithmic bytes, rows done, wall seconds)."""
    import oracle
    if x is None:
        x, _ = index_inputs()
    bits = x.view(torch.int16).numpy().view(np.uint16)
    rows, elapsed, i = 0, 0.0, 0
    while elapsed < budget_s and i < INDEX_TOKENS:
        chunks = [bits[j:j + 4096] for j in range(i, min(i + cores * 4096, INDEX_TOKENS), 4096)]
        elapsed += run_parallel([(lambda c=c: oracle.mxfp4_quantize_rows(c)) for c in chunks],
                                cores)
        n = sum(c.shape[0] for c in chunks)
        rows += n
        i += n
    return rows * INDEX_ROW_BYTES / elapsed / 1e9, rows, elapsed


def run_index(args, rank, local, world):
    import fp8_paged_kv_kvq_gb300 as kvq
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    K = args.steps if args.steps is not None else DEFAULT_STEPS["index"]
    W = max(3, args.warmup if args.warmup is not None else min(50, max(3, K // 10)))
    lib = kvq.load()
    x_h, slots_h = index_inputs()
    x, slots = x_h.to(dev), slots_h.to(dev)
    cache = kvq.IndexCache.empty(INDEX_TOKENS, kvq.INDEX_MXFP4, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)
    st = cache.struct()
    P = ctypes.c_void_p
    qargs = (ctypes.byref(st), P(x.data_ptr()), x.stride(0), INDEX_TOKENS, P(slots.data_ptr()),
             P(err.data_ptr()), P(stream.cuda_stream))

    def quantize():
        status = lib.kvq_index_quantize_scatter(*qargs)
        if status:
            raise RuntimeError(f"kvq_index_quantize_scatter: status {status}")

    with torch.cuda.stream(stream):
        quantize()
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            quantize()
        torch.cuda.synchronize(dev)
        flush = None if args.profile else L2Flush(dev)
        for i in range(W):
            if flush is not None:
                flush(i)
            graph.replay()
        torch.cuda.synchronize(dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
        sampler = ClockSampler(local) if not args.profile else None
        dist_barrier(world)
        torch.cuda.synchronize(dev)
        if sampler:
            sampler.start()
        wall0 = time.perf_counter()
        torch.cuda.nvtx.range_push("kvq_timed")
        for i in range(K):
            if flush is not None:
                flush(i + 7)
            evs[i][0].record(stream)
            graph.replay()
            evs[i][1].record(stream)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize(dev)
        wall1 = time.perf_counter()
        if sampler:
            sampler.stop()
        dist_barrier(world)
        ms = dist_max(sum(a.elapsed_time(b) for a, b in evs) / K, world)
        if int(err.item()) != 0:
            raise RuntimeError("device error flags set during the benchmark")
        peak, peak_src = measured_peaks()
        step_bytes = INDEX_TOKENS * INDEX_ROW_BYTES
        value = world * step_bytes / (ms * 1e-3) / 1e9
        res = {
            "metric": INDEX_METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": round(ms, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": DESCRIPTIONS["index"], "name": "index",
                       "l2": ("flushed before every timed step (256 MiB write, then a 256 MiB "
                              "read)") if flush is not None else "not flushed (profile mode)",
                       "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                       "storage": "E2M1 codes two per byte + an E8M0 exponent per 32 dims"},
            "pct_of_8tbs": round(100.0 * value / world / NOMINAL_HBM_GBS, 2),
            "pct_of_hbm_peak": round(100.0 * value / world / peak, 2),
            "rows_quantized_per_s": round(world * INDEX_TOKENS / (ms * 1e-3), 1),
            "kernels_us": {"index_quantize_scatter": round(1e3 * ms, 3)},
            "gpu_launches": K,
            "wall_s_timed_region": round(wall1 - wall0, 3),
        }
        achieved = step_bytes / (ms * 1e-3) / 1e9
        res["roofline"] = {
            "kernel": "index_quantize_kernel", "bound": "hbm", "achieved": round(achieved, 2),
            "peak": peak,
            "peak_source": ("measured (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                            else "fallback 6.8 TB/s"),
            "unit": "GB/s", "frac": round(achieved / peak, 4),
            "algorithmic_bytes_per_launch": step_bytes,
            "traffic": ncu_traffic("index_quantize_kernel", "index",
                                   "fp8_paged_kv_kvq_gb300/csrc/kvq_quantize.cu"),
        }
        if sampler:
            res["clocks"] = sampler.summary(wall0, wall1)
        if not args.profile and not args.no_e2e:
            xp = x_h.pin_memory()
            sp = slots_h.pin_memory()
            ep = torch.empty(cache.exponents.shape, dtype=torch.uint8, pin_memory=True)

            def body():
                x.copy_(xp, non_blocking=True)
                slots.copy_(sp, non_blocking=True)
                quantize()
                ep.copy_(cache.exponents, non_blocking=True)

            for _ in range(3):
                body()
            torch.cuda.synchronize(dev)
            n_e2e = max(20, min(K, 300))
            ems = dist_max(_timed(stream, dev, n_e2e, body, L2Flush(dev)), world)
            res["e2e"] = {"value": round(world * step_bytes / (ems * 1e-3) / 1e9, 2),
                          "unit": "GB/s", "ms_per_step": round(ems, 5),
                          "h2d_bytes_per_step": x_h.numel() * 2 + slots_h.numel() * 8,
                          "d2h_bytes_per_step": ep.numel()}
        if rank == 0 and world == 1 and not args.profile and not args.no_cpu_baseline:
            v1, rows1, secs1 = index_oracle_rate(6.0, x_h)
            cores = host_cores()
            v, rows, secs = index_oracle_rate(6.0, x_h, cores)
            res["cpu_baseline"] = {"value": round(v, 5), "unit": "GB/s", "cores": cores,
                                   "kind": "oracle",
                                   "sample": f"{rows} rows of the workload in 4096-row chunks "
                                             f"on {cores} host threads, {secs:.1f} s wall; one "
                                             f"thread: {rows1} rows in {secs1:.1f} s",
                                   "single_thread": {"value": round(v1, 5), "unit": "GB/s",
                                                     "cores": 1}}
    return res


def run_index_reference(args, rank, world):
    """--impl reference for the index workload: the oracle on the host."""
    if rank != 0:
        return None
    K = args.steps if args.steps is not None else 60
    W = max(3, args.warmup if args.warmup is not None else 3)
    budget = min(2.0, 150.0 / (K + W))
    x, _ = index_inputs()
    cores = host_cores()
    for _ in range(W):
        index_oracle_rate(budget / 4, x, cores)
    total_b, total_t = 0.0, 0.0
    for _ in range(K):
        _, rows, secs = index_oracle_rate(budget, x, cores)
        total_b += rows * INDEX_ROW_BYTES
        total_t += secs
    value = total_b / total_t / 1e9
    return {
        "impl": "reference", "metric": INDEX_METRIC, "value": round(value, 5), "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": round(1e3 * total_t / K, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": DESCRIPTIONS["index"], "name": "index"},
        "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"each step a bounded run of 4096-row chunks of the workload, "
                                   f"{cores} chunks at a time on {cores} host threads"},
        "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


# ---------------------------------------------------------------------------
# stacked index scores over MXFP4 index keys

SCORES_METRIC = ("stacked index scores over {} keys: achieved HBM GB/s (% of 8 TB/s); "
                 "tokens scored/s")


def scores_inputs(fmt: int = 1):
    """Host inputs of the index-scoring workload: block tables, context
    lengths, key codes with their scales (FP8, fmt 0) or exponents (MXFP4,
    fmt 1), bf16 queries [N, R, H, 128]."""
    import workloads
    w = workloads.INDEX_SCORES
    lens = np.full(w.num_requests, w.context, dtype=np.int32)
    bt, nblk = workloads.block_tables(lens, w.block_size, w.seed)
    codes, scales, exps = workloads.index_key_codes(fmt, nblk * w.block_size, w.seed)
    q = workloads.index_queries(w.num_requests, w.rows, w.heads, w.seed)
    return w, fmt, lens, bt, codes, scales, exps, q


def scores_step_bytes(w, fmt: int = 1) -> int:
    """Algorithmic bytes of one launch: every key read once (MXFP4: 64 code
    bytes + 4 exponent bytes per token; FP8: 128 + a 4-byte scale), the block
    tables, lengths and queries, and the fp32 scores of every (row, token)."""
    T = w.num_requests * w.context
    key = 64 + 4 if fmt == 1 else 128 + 4
    return (T * key + w.num_requests * (w.context // w.block_size) * 4 +
            w.num_requests * 4 + w.num_requests * w.rows * w.heads * 128 * 2 +
            w.num_requests * w.rows * w.context * 4)


def scores_oracle_rate(budget_s: float, inp=None, cores: int = 1):
    """The oracle's index scorer over whole requests of the workload, `cores`
    requests at a time on as many host threads, until the budget is spent:
    (tokens/s, requests done, wall seconds)."""
    import oracle
    w, fmt, lens, bt, codes, scales, exps, q = inp if inp is not None else scores_inputs()
    qb = q.view(torch.int16).numpy().view(np.uint16)
    done, elapsed = 0, 0.0
    while elapsed < budget_s and done < w.num_requests:
        rs = list(range(done, min(done + cores, w.num_requests)))
        elapsed += run_parallel(
            [(lambda r=r: oracle.index_scores(fmt, codes, scales, exps, bt[r:r + 1],
                                              w.block_size, lens[r:r + 1], w.rows, w.heads,
                                              qb[r].reshape(-1, 128), w.context))
             for r in rs], cores)
        done += len(rs)
    return done * w.context / elapsed, done, elapsed


def run_scores(args, rank, local, world):
    import fp8_paged_kv_kvq_gb300 as kvq
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    K = args.steps if args.steps is not None else DEFAULT_STEPS["scores"]
    W = max(3, args.warmup if args.warmup is not None else min(50, max(3, K // 10)))
    lib = kvq.load()
    fmt = 1 if args.index_format == "mxfp4" else 0
    inp = scores_inputs(fmt)
    w, _, lens_h, bt_h, codes_h, scales_h, exps_h, q_h = inp
    N = w.num_requests if args.requests <= 0 else min(args.requests, w.num_requests)
    cache = kvq.IndexCache.empty(codes_h.shape[0], fmt, device=dev)
    cache.codes.copy_(torch.from_numpy(codes_h))
    if fmt == 1:
        cache.exponents.copy_(torch.from_numpy(exps_h))
    else:
        cache.scales.copy_(torch.from_numpy(scales_h))
    bt = torch.from_numpy(bt_h[:N]).contiguous().to(dev)
    lens = torch.from_numpy(lens_h[:N]).to(dev)
    q = q_h[:N].contiguous().to(dev)
    out = torch.empty((N * w.rows, w.context), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)
    st = cache.struct()
    P = ctypes.c_void_p
    sargs = (ctypes.byref(st), w.block_size, P(q.data_ptr()), N, w.rows, w.heads,
             P(bt.data_ptr()), bt.shape[1], P(lens.data_ptr()), w.context, P(out.data_ptr()),
             P(err.data_ptr()), P(stream.cuda_stream))

    def score():
        status = lib.kvq_index_scores(*sargs)
        if status:
            raise RuntimeError(f"kvq_index_scores: status {status}")

    wN = dataclasses.replace(w, num_requests=N)
    step_bytes = scores_step_bytes(wN, fmt)
    fmt_name = "MXFP4" if fmt == 1 else "FP8"
    res = {}
    with torch.cuda.stream(stream):
        score()
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            score()
        torch.cuda.synchronize(dev)
        flush = None if args.profile else L2Flush(dev)
        for i in range(W):
            if flush is not None:
                flush(i)
            graph.replay()
        torch.cuda.synchronize(dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
        sampler = ClockSampler(local) if not args.profile else None
        dist_barrier(world)
        torch.cuda.synchronize(dev)
        if sampler:
            sampler.start()
        wall0 = time.perf_counter()
        torch.cuda.nvtx.range_push("kvq_timed")
        for i in range(K):
            if flush is not None:
                flush(i + 7)
            evs[i][0].record(stream)
            graph.replay()
            evs[i][1].record(stream)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize(dev)
        wall1 = time.perf_counter()
        if sampler:
            sampler.stop()
        dist_barrier(world)
        ms = dist_max(sum(a.elapsed_time(b) for a, b in evs) / K, world)
        if int(err.item()) != 0:
            raise RuntimeError("device error flags set during the benchmark")
        peak, peak_src = measured_peaks()
        value = world * step_bytes / (ms * 1e-3) / 1e9
        tokens = N * w.context
        res = {
            "metric": SCORES_METRIC.format(fmt_name), "value": round(value, 2), "unit": "GB/s",
            "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": round(ms, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": DESCRIPTIONS["scores"].replace("MXFP4", fmt_name),
                       "name": "scores", "requests": N,
                       "l2": ("flushed before every timed step (256 MiB write, then a 256 MiB "
                              "read)") if flush is not None else "not flushed (profile mode)",
                       "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                       "keys": ("E2M1 codes two per byte + an E8M0 exponent per 32 dims"
                                if fmt == 1 else "e4m3 codes + fp32 scale per row") +
                               ", random codes"},
            "pct_of_8tbs": round(100.0 * value / world / NOMINAL_HBM_GBS, 2),
            "pct_of_hbm_peak": round(100.0 * value / world / peak, 2),
            "tokens_scored_per_s": round(world * tokens / (ms * 1e-3), 1),
            "kernels_us": {"index_scores": round(1e3 * ms, 3)},
            "gpu_launches": K,
            "wall_s_timed_region": round(wall1 - wall0, 3),
        }
        achieved = step_bytes / (ms * 1e-3) / 1e9
        res["roofline"] = {
            "kernel": "index_scores_kernel", "bound": "hbm", "achieved": round(achieved, 2),
            "peak": peak,
            "peak_source": ("measured (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                            else "fallback 6.8 TB/s"),
            "unit": "GB/s", "frac": round(achieved / peak, 4),
            "algorithmic_bytes_per_launch": step_bytes,
            "traffic": ncu_traffic("index_scores_kernel", "scores",
                                   "fp8_paged_kv_kvq_gb300/csrc/kvq_index_scores.cu"),
        }
        if sampler:
            res["clocks"] = sampler.summary(wall0, wall1)
        if not args.profile and not args.no_e2e:
            qp = torch.empty(q.shape, dtype=q.dtype, pin_memory=True).copy_(q_h[:N])
            btp = torch.empty(bt.shape, dtype=bt.dtype, pin_memory=True).copy_(
                torch.from_numpy(bt_h[:N]))
            lp = torch.empty(lens.shape, dtype=lens.dtype, pin_memory=True).copy_(
                torch.from_numpy(lens_h[:N]))
            op = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)

            def body():
                q.copy_(qp, non_blocking=True)
                bt.copy_(btp, non_blocking=True)
                lens.copy_(lp, non_blocking=True)
                score()
                op.copy_(out, non_blocking=True)

            for _ in range(3):
                body()
            torch.cuda.synchronize(dev)
            n_e2e = max(20, min(K, 200))
            ems = dist_max(_timed(stream, dev, n_e2e, body, L2Flush(dev)), world)
            res["e2e"] = {"value": round(world * step_bytes / (ems * 1e-3) / 1e9, 2),
                          "unit": "GB/s", "ms_per_step": round(ems, 5),
                          "h2d_bytes_per_step": sum(t.numel() * t.element_size()
                                                    for t in (qp, btp, lp)),
                          "d2h_bytes_per_step": op.numel() * op.element_size()}
        if rank == 0 and world == 1 and not args.profile and not args.no_cpu_baseline:
            tps1, done1, secs1 = scores_oracle_rate(6.0, inp)
            cores = host_cores()
            tps, done, secs = scores_oracle_rate(6.0, inp, cores)
            res["cpu_baseline"] = {"value": round(tps * step_bytes / tokens / 1e9, 5),
                                   "unit": "GB/s", "cores": cores, "kind": "oracle",
                                   "tokens_per_s": round(tps, 1),
                                   "sample": f"{done} whole requests of the workload, {cores} "
                                             f"at a time on {cores} host threads, {secs:.1f} s "
                                             f"wall; one thread: {done1} requests in "
                                             f"{secs1:.1f} s",
                                   "single_thread": {"value": round(tps1 * step_bytes / tokens
                                                                    / 1e9, 5),
                                                     "unit": "GB/s", "cores": 1}}
    return res


def run_scores_reference(args, rank, world):
    """--impl reference for the index-scoring workload: the oracle on the host."""
    if rank != 0:
        return None
    K = args.steps if args.steps is not None else 40
    W = max(3, args.warmup if args.warmup is not None else 3)
    budget = min(2.5, 150.0 / (K + W))
    fmt = 1 if args.index_format == "mxfp4" else 0
    fmt_name = "MXFP4" if fmt == 1 else "FP8"
    inp = scores_inputs(fmt)
    w = inp[0]
    per_token = scores_step_bytes(w, fmt) / (w.num_requests * w.context)
    cores = host_cores()
    for _ in range(W):
        scores_oracle_rate(budget / 4, inp, cores)
    total_tok, total_t = 0.0, 0.0
    for _ in range(K):
        _, done, secs = scores_oracle_rate(budget, inp, cores)
        total_tok += done * w.context
        total_t += secs
    value = total_tok * per_token / total_t / 1e9
    return {
        "impl": "reference", "metric": SCORES_METRIC.format(fmt_name), "value": round(value, 5),
        "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": round(1e3 * total_t / K, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": DESCRIPTIONS["scores"].replace("MXFP4", fmt_name), "name": "scores"},
        "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"each step whole requests of the workload, {cores} at a "
                                   f"time on {cores} host threads, until a bounded time is "
                                   f"spent"},
        "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main(argv=None):
    args = parse_args(argv)
    rank, local, world = dist_init()
    if args.workload == "scores":
        res = run_scores_reference(args, rank, world) if args.impl == "reference" else \
            run_scores(args, rank, local, world)
    elif args.workload == "index":
        res = run_index_reference(args, rank, world) if args.impl == "reference" else \
            run_index(args, rank, local, world)
    else:
        res = run_reference(args, rank, world) if args.impl == "reference" else \
            run_kvq(args, rank, local, world)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
