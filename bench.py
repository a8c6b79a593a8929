"""Benchmark: one decode step of paged attention on GB300.

A step is the whole hot path over one batch: copy-on-write block copies (none
in this workload), then the slot write of the step's new K/V and decode
attention through the block tables (with its split-K merge), one fused launch
(pkv_decode_step).  The default workload is the
Qwen2.5-7B-shaped layer in bf16: 28 query / 4 KV heads, head_dim 128, block
16, pool 8,500 blocks, 64 sequences with contexts uniform on [256, 4096].

Prints one JSON line.  ``value`` is the attention's algorithmic K/V bytes
(every cached K/V element once) divided by the device time of the step, in
GB/s, inputs resident in HBM and larger than L2, the K timed steps replayed
back to back from one CUDA graph; ``e2e`` is
the same metric through the C ABI with the step's inputs copied from pinned
host memory and the output copied back inside the timed region.  With
``--impl reference`` the CPU oracle is timed on the host instead.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import shutil
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_CONFIG = "qwen_gqa_bf16"
# the other decode workloads the default run also measures (``per_config``)
OTHER_CONFIGS = ("tiny_fp32", "prefix_fork_bf16", "long_mha_bf16", "fp8_churn")
METRIC = "paged decode attention KV GB/s & fraction of GB300 HBM peak; decode tokens/s"
# the sources each kernel family's recorded DRAM counters depend on
KERNEL_SOURCES = {
    "decode": ["attention.cu", "attention.h", "attention_simt.cuh", "attention_tc.cuh",
               "attention_tc_launch.cuh", "device_common.cuh", "attention_prefill_umma.cuh",
               "attention_shared_prefix.cu", "attention_tail.cuh"],
    "prefill": ["attention_prefill.cu", "attention_prefill_umma.cuh", "attention_tc.cuh", "attention.h",
                "device_common.cuh"],
}
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-per-config", action="store_true",
                    help="measure only the configured workload (default: also the other decode "
                         "workloads, under per_config)")
    ap.add_argument("--per-config-cpu-seconds", type=float, default=3.0)
    ap.add_argument("--timed-ms", type=float, default=200.0,
                    help="device time each timed graph is replayed for, at least (0: five replays "
                         "and K end-to-end steps, for profiling runs)")
    ap.add_argument("--partition", type=int, default=None,
                    help="split-K partition in tokens (default: the workload's, else automatic)")
    ap.add_argument("--kernel", default="auto", choices=["auto", "simt", "tc"],
                    help="decode kernel (auto = tensor-core where it applies)")
    ap.add_argument("--shared-prefix", default="auto", choices=["auto", "on", "off"],
                    help="decode a batch's shared prefix once for all sequences (auto: when the "
                         "batch shares at least 256 tokens over at least 128 query rows)")
    ap.add_argument("--block-size", type=int, default=None,
                    help="ablation: tokens per block (the pool keeps the same token capacity)")
    ap.add_argument("--fp8-scales", default="tensor", choices=["tensor", "head"],
                    help="ablation: E4M3 scales per tensor or per KV head")
    ap.add_argument("--kv-dtype", default=None, choices=["bf16", "f16", "e4m3"],
                    help="ablation: cache dtype (q stays 16-bit)")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def code_only(text: str) -> str:
    """A C++/CUDA source without its comments and blank lines: what the
    compiler sees (the sources hold no string literal with a comment marker),
    so that editing a comment does not retire the counters taken on the code."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash(family: str = "decode") -> str:
    h = hashlib.sha256()
    for n in KERNEL_SOURCES[family]:
        with open(os.path.join(ROOT, "paged_kv_cache_137_gb300", "csrc", n)) as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def allocator_step_us(plan, steps: int = 200) -> float:
    """Host time of one decode step of the native allocator for the plan's
    batch: pkv_batch_append of one token per sequence, then
    pkv_block_tables_update of the batch's tables kept across steps (a fresh
    pool replaying the plan's prefill)."""
    import numpy as np
    import paged_kv_cache_137_gb300 as pkv
    w = plan.w
    t = w.block_size
    # private blocks for every sequence (a forked plan's shared prefix is
    # replayed per sequence), plus room for the timed appends
    need = sum(-(-int(c) // t) for c in plan.ctx) + len(plan.seq_ids) * (steps // t + 2)
    pool = pkv.Pool(max(w.num_blocks, need), t)
    for s, c in zip(plan.seq_ids, plan.ctx):
        pool.seq_create(s)
        pool.seq_append(s, int(c))
    max_blocks = plan.max_blocks + steps // w.block_size + 2
    # the batch's tables kept in host buffers across steps and brought up to
    # date incrementally, as a serving loop that stages them for one copy to
    # the device would
    ids = np.asarray(plan.seq_ids, dtype=np.int64)
    rows = pool.block_tables_rows(len(ids), max_blocks)
    rows.update(ids)
    t0 = time.perf_counter()
    for _ in range(steps):
        pool.batch_append(ids)
        rows.update(ids)
    return (time.perf_counter() - t0) / steps * 1e6


def e2e_graph_of(e2e_step, dev_in, host_in, scn, out_host, steps: int, kv_bytes: int):
    """The end-to-end step (host-to-device copy of the inputs, the step, the
    device-to-host copy of the output) captured as ONE CUDA graph and
    replayed once per step with a host synchronisation after each, as a
    serving loop that replays a captured step would: GB/s over the host's
    wall clock.  Reported beside the eager end-to-end figure; a capture that
    the installed PyTorch refuses is reported as such."""
    import torch
    try:
        e2e_step()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            dev_in.copy_(host_in, non_blocking=True)
            scn.step()
            out_host.copy_(scn.out, non_blocking=True)
        for _ in range(3):
            g.replay()
            torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(steps):
            g.replay()
            torch.cuda.synchronize()
        s = (time.perf_counter() - t0) / steps
    except RuntimeError as e:
        return {"error": str(e).splitlines()[0][:200]}
    return {"value": round(kv_bytes / s / 1e9, 2), "unit": "GB/s", "ms_per_step": round(s * 1e3, 4),
            "what": "copy in, step, copy out captured as one CUDA graph, one replay and one host "
                    "sync per step"}


def packed(tensors, device):
    """One device buffer holding the given tensors back to back (each at a
    256-byte boundary), so that a step's inputs arrive by ONE host-to-device
    copy: the buffer and views of it holding the tensors' values."""
    import torch
    offs, total = [], 0
    for t in tensors:
        offs.append(total)
        total += -(-t.numel() * t.element_size() // 256) * 256
    buf = torch.zeros(total, dtype=torch.uint8, device=device)
    views = []
    for t, o in zip(tensors, offs):
        v = buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
        v.copy_(t)
        views.append(v)
    return buf, views


def workload_of(args):
    """The configured workload, with the ablation overrides applied: another
    block size keeps the pool's token capacity (plus one block per sequence,
    so that the same context lengths are drawn), another cache dtype keeps
    the shapes."""
    import workloads as W
    w = W.get(args.config)
    if args.block_size and args.block_size != w.block_size:
        nb = -(-w.num_blocks * w.block_size // args.block_size) + w.num_seqs
        w = W.scaled(w, block_size=args.block_size, num_blocks=nb)
    if args.kv_dtype and args.kv_dtype != w.kv_dtype:
        q = w.q_dtype if args.kv_dtype == "e4m3" else args.kv_dtype
        w = W.scaled(w, kv_dtype=args.kv_dtype, q_dtype="bf16" if q == "f32" else q)
    return w


def attention_kernels(kernel: str, w, splits: int, shared_prefix: bool = False) -> str:
    """The kernels one attention call launches (timed together, as one graph)."""
    if w.kv_dtype == "f32" or kernel == "simt":
        k = "decode_simt_kernel"
        return k + (" + merge_kernel" if splits > 1 else "")
    if shared_prefix:
        # the tail queue: 16-bit caches, head_dim 128, block size 16, groups of
        # up to 8 and a unit list of at most 512 sequences (else the split
        # kernel's narrow forms)
        queue = (kernel == "auto" and w.kv_dtype in ("bf16", "f16") and w.block_size == 16 and
                 w.head_dim == 128 and w.num_q_heads // w.num_kv_heads <= 8 and w.num_seqs <= 512)
        tails = "tail_stream_kernel" if queue else "decode_tc_kernel"
        return f"prefill_umma_kernel<shared prefix> + {tails} + prefix_merge_kernel"
    return "decode_tc_kernel (split-K merge fused)"


def traffic_for(config: str, kernels: str):
    """DRAM bytes per attention launch from the committed ncu summary, if it
    was taken on the current kernel sources and the same kernel."""
    p = os.path.join(ROOT, "profiles", "attention_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get(config)
    family = e.get("family", "decode") if e else "decode"
    if not e or e.get("kernel_sha") != kernel_source_hash(family):
        return None
    if not kernels.startswith(e.get("kernel", "?").split("<")[0]):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """SM clock and throttle reasons sampled through NVML (ctypes, read-only)
    every ~0.5 ms while the timed region runs; nvidia-smi when NVML is absent."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    SMI_QUERY = "clocks.sm,clocks.max.sm,clocks_event_reasons.active"

    def __init__(self, index: int):
        import ctypes
        self.index = index
        self.samples, self.max_mhz, self.stop = [], None, threading.Event()
        self.nvml, self.smi = None, None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            h = ctypes.c_void_p()
            if nv.nvmlInit_v2() == 0 and nv.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(h)) == 0:
                self.nvml, self.handle = nv, h
                mx = ctypes.c_uint()
                if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                    self.max_mhz = float(mx.value)
                fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                    nv.nvmlDeviceGetCurrentClocksThrottleReasons
                self.reasons_fn = fn
        except OSError:
            self.nvml = None

    def _poll(self):
        import ctypes
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk)) == 0 and \
                    self.reasons_fn(self.handle, ctypes.byref(rs)) == 0:
                self.samples.append((float(clk.value), int(rs.value)))
            time.sleep(0.0005)

    @staticmethod
    def parse_smi(text: str):
        """Samples from `nvidia-smi --query-gpu=<SMI_QUERY> --format=csv,noheader,nounits`
        lines: [(sm MHz, reasons bitmask)] and the max SM clock (None if absent)."""
        samples, mx = [], None
        for line in text.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) != 3:
                continue
            try:
                clk, top, rs = float(f[0]), float(f[1]), int(f[2], 16)
            except ValueError:
                continue
            samples.append((clk, rs))
            mx = top
        return samples, mx

    def __enter__(self):
        if self.nvml is not None:
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
        elif shutil.which("nvidia-smi"):
            # read-only query of this GPU every 200 ms, stopped in __exit__
            self.smi = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.SMI_QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        return self

    def __exit__(self, *exc):
        self.stop.set()
        if self.nvml is not None:
            self.thread.join(timeout=2)
        elif self.smi is not None:
            self.smi.terminate()
            try:
                out, _ = self.smi.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.smi.kill()
                out, _ = self.smi.communicate()
            self.samples, self.max_mhz = self.parse_smi(out or "")

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"], "samples": 0}
        reasons = sorted({name for _, r in self.samples for bit, name in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(c for c, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.samples),
                "source": "nvml" if self.nvml is not None else "nvidia-smi"}


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if args.impl == "gb300":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
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
    device = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ oracle
class OracleRunner:
    """The CPU oracle on the host.  One pass = decode attention of the whole
    batch of the workload over the oracle's pool (built once, not timed)."""

    def __init__(self, config: str):
        import numpy as np
        import workloads as W
        from oracle import scenario as OS
        self.w = w = W.get(config)
        self.sc = W.fp8_scales(*W.kv_amax(w)) if w.kv_dtype == "e4m3" else {}
        self.scn = OS.build(w, scales=self.sc)
        self.q = self.scn.q_f64()
        self.tables = self.scn.tables
        self.kv_bytes = 2 * int(np.sum(self.scn.ctx)) * w.num_kv_heads * w.head_dim * w.kv_bytes

    def one_pass(self) -> float:
        import math
        from oracle import attention as OA
        t0 = time.perf_counter()
        OA.paged_attention_decode(self.q, self.scn.pool, self.tables, self.scn.ctx,
                                  1.0 / math.sqrt(self.w.head_dim), self.sc.get("k_scale", 1.0),
                                  self.sc.get("v_scale", 1.0))
        return time.perf_counter() - t0

    def timed(self, seconds: float):
        """Passes until ``seconds`` elapse -> (GB/s, passes, elapsed)."""
        el, passes = 0.0, 0
        while passes == 0 or el < seconds:
            el += self.one_pass()
            passes += 1
        return self.kv_bytes * passes / el / 1e9, passes, el


# ---- the oracle on all host cores: a spawn-context process pool whose
# workers each hold the oracle's pool and compute the decode attention of an
# interleaved share of the batch's sequences (the oracle function unchanged;
# one BLAS thread per worker)
_POOL_RUNNER = None


def _pool_init(config: str):
    import workloads as W
    global _POOL_RUNNER
    w = W.get(config)
    _POOL_RUNNER = PrefillOracle(config, w.num_seqs) if w.prefill_chunk else OracleRunner(config)


def _pool_rows(rows) -> float:
    import math
    r = _POOL_RUNNER
    t0 = time.perf_counter()
    if isinstance(r, PrefillOracle):
        from oracle import prefill as OP
        OP.paged_attention_prefill(r.q, r.scn.pool, r.scn.tables, r.scn.ctx, r.qs,
                                   1.0 / math.sqrt(r.w.head_dim), seqs=rows)
    else:
        from oracle import attention as OA
        OA.paged_attention_decode(r.q, r.scn.pool, r.tables, r.scn.ctx, 1.0 / math.sqrt(r.w.head_dim),
                                  r.sc.get("k_scale", 1.0), r.sc.get("v_scale", 1.0), seqs=rows)
    return time.perf_counter() - t0


class OraclePool:
    """The oracle's whole-batch decode (or, for a prefill workload, prefill)
    attention spread over worker processes (spawn context, one BLAS thread
    each), sequences interleaved over the workers; the pool's set-up is not
    timed.  ``units`` is the work of one pass: K/V bytes, or FLOPs."""

    def __init__(self, config: str, cores: int | None = None):
        import numpy as np
        import workloads as W
        self.w = w = W.get(config)
        ctx = W.context_lens(w) if w.ctx_dist != "prefix_fork" else W.fork_layout(w)["ctx"]
        self.kv_bytes = 2 * int(np.sum(ctx)) * w.num_kv_heads * w.head_dim * w.kv_bytes
        self.flops = prefill_flops(w, ctx, W.chunk_lens(w, ctx, w.prefill_chunk)) if w.prefill_chunk else 0
        self.units = self.flops if w.prefill_chunk else self.kv_bytes
        self.n = max(1, min(cores or len(os.sched_getaffinity(0)), w.num_seqs))
        self.chunks = [list(range(i, w.num_seqs, self.n)) for i in range(self.n)]
        import multiprocessing as mp
        saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"
        try:
            self.pool = mp.get_context("spawn").Pool(self.n, initializer=_pool_init, initargs=(config,))
            self.pool.map(_pool_rows, self.chunks)  # every worker built and warm
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def one_pass(self) -> float:
        t0 = time.perf_counter()
        self.pool.map(_pool_rows, self.chunks)
        return time.perf_counter() - t0

    def one_core_pass(self) -> float:
        return self.pool.apply(_pool_rows, (list(range(self.w.num_seqs)),))

    def close(self):
        self.pool.close()
        self.pool.join()


def parallel_oracle(config: str, seconds: float, cores: int | None = None):
    """Whole-batch passes on all workers until ``seconds`` elapse, then one
    on one worker -> (rate, passes, elapsed, workers, rate on one core); the
    rate is GB/s for decode, TFLOP/s for prefill."""
    p = OraclePool(config, cores)
    try:
        el, passes = 0.0, 0
        while passes == 0 or el < seconds:
            el += p.one_pass()
            passes += 1
        one = p.one_core_pass()
    finally:
        p.close()
    scale = 1e12 if p.flops else 1e9
    return p.units * passes / el / scale, passes, el, p.n, p.units / one / scale


def run_reference(args, world, rank):
    if rank != 0:
        return
    r = OraclePool(args.config)
    try:
        for _ in range(args.warmup):
            r.one_pass()
        t_steps = [r.one_pass() for _ in range(args.steps)]
    finally:
        r.close()
    ms = 1e3 * statistics.mean(t_steps)
    gbs = r.kv_bytes / (ms / 1e3) / 1e9
    w = r.w
    sample = (f"whole batch of {args.config} ({w.num_seqs} sequences), one pass per step "
              f"on {r.n} worker processes")
    line = {"metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": args.config, "num_seqs": w.num_seqs, "kv_bytes_per_step": r.kv_bytes},
            "tokens_per_s": round(w.num_seqs / (ms / 1e3), 3),
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": r.n, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------- GPU
def replay_timed(graph, stream, min_ms: float, max_replays: int = 5000):
    """Replay a captured graph back to back until at least ``min_ms`` of
    device time is timed (the first replay sizes the count, at least 5),
    each replay bracketed by CUDA events on ``stream`` -> per-replay ms."""
    import torch
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    graph.replay()
    b.record(stream)
    torch.cuda.synchronize()
    n = int(min(max_replays, max(5, -(-min_ms // max(a.elapsed_time(b), 1e-3)))))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in evs:
        a.record(stream)
        graph.replay()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def capture(fn, K: int):
    """K calls of ``fn`` captured back to back in one CUDA graph."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(K):
            fn()
    g.replay()
    return g


def warm(scn, n: int, device):
    """n untimed steps on a side stream (the capture warm-up PyTorch asks for)."""
    import torch
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream(device=device)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for _ in range(n):
            scn.step()
    stream.wait_stream(side)
    torch.cuda.synchronize()


def scenario_for(config: str, args, device, w=None):
    import workloads as W
    from paged_kv_cache_137_gb300 import scenario as PS
    w = w or W.get(config)
    sc = {}
    if w.kv_dtype == "e4m3":
        sc = W.fp8_head_scales(w) if args.fp8_scales == "head" else W.fp8_scales(*W.kv_amax(w))
    return PS.materialize(PS.plan(w), device, sc, partition_tokens=args.partition,
                          shared_prefix={"auto": None, "on": True, "off": False}[args.shared_prefix])


def oracle_sample(config: str, seconds: float, n_rows: int = 4):
    """The oracle (unchanged) on one host core over a bounded sample of a
    workload: ``n_rows`` sequences spread over the batch (their pool blocks
    written, the rest of the batch only planned), passes until ``seconds``
    elapse -> cpu_baseline entry (GB/s of their logical K/V bytes)."""
    import math
    import numpy as np
    import workloads as W
    from oracle import attention as OA
    from oracle import scenario as OS
    w = W.get(config)
    sc = W.fp8_scales(*W.kv_amax(w)) if w.kv_dtype == "e4m3" else {}
    rows = sorted({int(r) for r in np.linspace(0, w.num_seqs - 1, min(n_rows, w.num_seqs))})
    scn = OS.build(w, write_seqs=rows, scales=sc)
    q = scn.q_f64()
    nbytes = 2 * int(np.sum(np.asarray(scn.ctx)[rows])) * w.num_kv_heads * w.head_dim * w.kv_bytes
    el, passes = 0.0, 0
    while passes == 0 or el < seconds:
        t0 = time.perf_counter()
        OA.paged_attention_decode(q, scn.pool, scn.tables, scn.ctx, 1.0 / math.sqrt(w.head_dim),
                                  sc.get("k_scale", 1.0), sc.get("v_scale", 1.0), seqs=rows)
        el += time.perf_counter() - t0
        passes += 1
    return {"value": round(nbytes * passes / el / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"sequences {rows} of {config} ({nbytes / 1e6:.1f} MB of K/V), {passes} pass(es) "
                      f"in {el:.1f} s on one host core"}


def per_config_entry(config: str, args, device, local, peak: float):
    """One workload's device figures (no reference arm, no end-to-end leg):
    the K-step graph and the K-attention graph each replayed for half of
    --timed-ms (100 ms by default),
    medians; the roofline over the distinct cache bytes; an oracle sample."""
    import numpy as np
    import torch
    scn = scenario_for(config, args, device)
    w = scn.plan.w
    stream = torch.cuda.current_stream()
    K = args.steps
    warm(scn, max(args.warmup, 3), device)
    g_steps, g_attns = capture(scn.step, K), capture(scn.attend, K)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        steps = replay_timed(g_steps, stream, args.timed_ms / 2)
        attns = replay_timed(g_attns, stream, args.timed_ms / 2)
    ms = statistics.median(steps) / K
    attn = statistics.median(attns) / K
    kv_bytes, unique = scn.kv_bytes(), scn.kv_unique_bytes()
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    kernels = attention_kernels(args.kernel, w, 2, bool(scn.prefix_blocks))
    traffic = traffic_for(config, kernels)
    e = {"workload": config, "num_seqs": w.num_seqs, "kv_dtype": w.kv_dtype,
         "kv_bytes_per_step": kv_bytes, "algorithmic_bytes": unique,
         "shared_prefix_blocks": scn.prefix_blocks, "partition_tokens": scn.partition,
         "ms_per_step": round(ms, 4), "value": round(kv_bytes / (ms / 1e3) / 1e9, 2), "unit": "GB/s",
         "tokens_per_s": round(w.num_seqs / (ms / 1e3), 1),
         "attention_ms": round(attn, 4), "kernel": kernels,
         "achieved": round(unique / (attn / 1e3) / 1e9, 2),
         "frac": round(unique / (attn / 1e3) / 1e9 / peak, 4),
         "traffic": traffic,
         **({"dram_achieved": round(traffic / (attn / 1e3) / 1e9, 2)} if traffic else {}),
         "replays": {"steps": len(steps), "attention": len(attns)},
         "l2": "inputs %s than L2 (distinct K/V %d MB vs %d MB)" % (
             "larger" if unique > l2 else "smaller", unique >> 20, l2 >> 20),
         "clocks": clk.summary()}
    if unique != kv_bytes:
        e["logical_achieved"] = round(kv_bytes / (attn / 1e3) / 1e9, 2)
    if w.kv_dtype == "f32":
        e["note"] = "correctness workload: too small to time meaningfully"
    del scn, g_steps, g_attns
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return e


def run_gpu(args, world, rank, local):
    import numpy as np
    import torch
    import workloads as W
    import paged_kv_cache_137_gb300 as pkv

    pkv.build()
    pkv.pkv_set_attention_kernel(args.kernel)
    torch.cuda.set_device(local)
    dev_name = f"cuda:{local}"
    w = workload_of(args)
    scn = scenario_for(args.config, args, dev_name, w)
    stream = torch.cuda.current_stream()
    kv_bytes = scn.kv_bytes()
    props = torch.cuda.get_device_properties(local)
    # L2 eviction for the isolated figures: a READ of a buffer twice the L2
    # size.  Writing it instead would leave the L2 full of dirty lines whose
    # write-back to HBM then competes with the step's own reads (about 10 %
    # of the attention time on this workload), a cost no decode step sees.
    flush = torch.ones(2 * props.L2_cache_size // 4 + 1024, dtype=torch.float32, device=dev_name)
    flush_sink = torch.empty((), dtype=torch.float32, device=dev_name)
    n_pairs = len(scn.plan.cow_pairs)
    resolved = pkv.pkv_attention_partition(len(scn.plan.seq_ids), scn.plan.max_blocks, scn.desc,
                                           scn.partition)
    splits = -(-scn.plan.max_blocks * w.block_size // resolved)
    # write + decode (+ the separate merge of the CUDA-core kernel) + block copies
    # the split-K merge is its own launch only in the CUDA-core path, and so
    # is the slot write outside the tensor-core split kernel (which fuses it)
    separate_merge = args.kernel == "simt" or w.kv_dtype == "f32"
    fused_write = not separate_merge
    # a shared prefix adds its pass before the decode kernel and the merge kernel after it
    attn_launches = 1 + (1 if separate_merge and splits > 1 else 0) + (2 if scn.prefix_blocks else 0)
    launches_per_step = (0 if fused_write else 1) + attn_launches + \
        (-(-n_pairs // 1024) if n_pairs else 0)

    warm(scn, max(args.warmup, 3), dev_name)
    # Timed region: the K steps (block copies, slot write, decode attention)
    # captured back to back in ONE CUDA graph, as a serving loop replays a
    # whole decode step: no library call and no graph launch sits between two
    # steps (one graph launch costs several microseconds on its own).  The
    # graph is replayed back to back until at least --timed-ms (200 ms) of device time is
    # timed, each replay between CUDA events; ms_per_step is the median
    # replay / K.  No L2 flush between steps: the K/V each step reads is
    # larger than the L2.  K attention calls in a second graph, timed the
    # same way (half as long), give the decode kernel's average duration for the
    # roofline.  The isolated figures (one step per graph launch, the L2
    # evicted by a read before each) are reported beside them.
    K = args.steps
    g_steps, g_attns = capture(scn.step, K), capture(scn.attend, K)
    torch.cuda.synchronize()

    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        step_reps = replay_timed(g_steps, stream, args.timed_ms)
        torch.cuda.synchronize()
        barrier(world)
        attn_reps = replay_timed(g_attns, stream, args.timed_ms / 2)
    ms = max_over_ranks(statistics.median(step_reps) / K, world)
    attn = statistics.median(attn_reps) / K
    value = world * kv_bytes / (ms / 1e3) / 1e9

    # isolated: one step (or one attention call) per graph launch, L2 evicted
    g_step, g_attn = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step):
        scn.step()
    with torch.cuda.graph(g_attn):
        scn.attend()
    iso = {"step": [], "attention": []}
    for _ in range(20):
        for name, g in (("step", g_step), ("attention", g_attn)):
            torch.sum(flush, dim=(0,), out=flush_sink)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            iso[name].append((a, b))
    torch.cuda.synchronize()
    iso_ms = {k: statistics.median(a.elapsed_time(b) for a, b in v) for k, v in iso.items()}

    # the step's small kernels: 20 calls captured in one graph, so the graph's
    # launch cost is spread over them (each call rewrites the same slots or
    # copies the same blocks)
    def per_call_us(fn, reps=20):
        g = capture(fn, reps)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / reps

    kvb = w.kv_bytes
    n_new = len(scn.plan.seq_ids) * w.num_kv_heads * w.head_dim
    write_bytes = 2 * n_new * (scn.k_new.element_size() + kvb) + 8 * len(scn.plan.seq_ids)
    write_us = per_call_us(scn.write_step)
    aux = {"slot_write_us": round(write_us, 2),
           "slot_write_GBs": round(write_bytes / (write_us * 1e3), 2),
           "copy_blocks_pairs": n_pairs}
    if n_pairs:
        copy_us = per_call_us(scn.copy_blocks)
        block_bytes = w.num_kv_heads * w.block_size * w.head_dim * kvb
        aux["copy_blocks_us"] = round(copy_us, 2)
        aux["copy_blocks_GBs"] = round(2 * 2 * n_pairs * block_bytes / (copy_us * 1e3), 2)

    # the host allocator's step (native C++): one token appended to each of the
    # batch's sequences and their block tables exported, on a copy of the plan
    aux["allocator_step_us"] = round(allocator_step_us(scn.plan), 2)

    e2e, e2e_graph = end_to_end(scn, dev_name, K if args.timed_ms == 0 else max(K, 200), world, kv_bytes)

    peak, peak_kind = peaks()
    kernels = attention_kernels(args.kernel, w, splits, bool(scn.prefix_blocks))
    # the profiled counters describe the configured workload only
    traffic = traffic_for(args.config, kernels) if w == W.get(args.config) else None
    # the roofline's algorithmic bytes: each stored K/V element once, however
    # many sequences share its block (the logical bytes where none is shared)
    unique_bytes = scn.kv_unique_bytes()
    achieved = unique_bytes / (attn / 1e3) / 1e9
    shared = {}
    if unique_bytes != kv_bytes:
        shared = {"algorithmic_bytes": unique_bytes,
                  "logical_achieved": round(kv_bytes / (attn / 1e3) / 1e9, 2),
                  "note": "blocks shared by several sequences count once in achieved"}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": max(args.warmup, 3), "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.kv_dtype == "bf16" else w.kv_dtype,
        "data": "synthetic",
        "config": {"workload": args.config, "num_seqs": w.num_seqs, "num_q_heads": w.num_q_heads,
                   "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
                   "num_blocks": w.num_blocks, "context_tokens": int(scn.plan.ctx.sum()),
                   "kv_bytes_per_step": kv_bytes, "partition_tokens": scn.partition,
                   "shared_prefix_blocks": scn.prefix_blocks,
                   "kv_dtype": w.kv_dtype, "table_entries": int(np.ceil(scn.plan.ctx / w.block_size).sum()),
                   **({"fp8_scales": args.fp8_scales} if w.kv_dtype == "e4m3" else {}),
                   "waste_slots_per_seq": round(float((np.ceil(scn.plan.ctx / w.block_size) * w.block_size
                                                       - scn.plan.ctx).mean()), 2),
                   "l2": ("inputs larger than L2 (K/V %d MB vs %d MB L2), no flush between steps"
                          % (kv_bytes >> 20, props.L2_cache_size >> 20)),
                   "launch": ("the K steps captured back to back in one CUDA graph; the graph replayed "
                              "%d times back to back (%.0f ms timed), median replay / K"
                              % (len(step_reps), sum(step_reps))),
                   "parallelism": "replicas" if world > 1 else "single"},
        "tokens_per_s": round(world * w.num_seqs / (ms / 1e3), 1),
        "frac_of_hbm_peak": round(value / peak, 4),
        "frac_of_nominal_hbm": round(value / NOMINAL_HBM_GBS, 4),
        "roofline": {"bound": "hbm", "kernel": kernels,
                     "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                     "traffic": traffic, "attention_ms": round(attn, 4),
                     "attention_replays": len(attn_reps),
                     **({"dram_achieved": round(traffic / (attn / 1e3) / 1e9, 2)} if traffic else {}),
                     **shared},
        "e2e": e2e,
        **({"e2e_graph": e2e_graph} if e2e_graph is not None else {}),
        "gpu_launches": (len(step_reps) + 1) * K * launches_per_step
                        + (len(attn_reps) + 1) * K * attn_launches,
        "aux": aux,
        "isolated": {"what": "one step (one attention call) per graph launch, L2 evicted by reading a "
                             "2x-L2 buffer before each; median of 20",
                     "step_ms": round(iso_ms["step"], 4), "attention_ms": round(iso_ms["attention"], 4),
                     "value": round(world * kv_bytes / (iso_ms["step"] / 1e3) / 1e9, 2),
                     "attention_GBs": round(unique_bytes / (iso_ms["attention"] / 1e3) / 1e9, 2),
                     "attention_frac": round(unique_bytes / (iso_ms["attention"] / 1e3) / 1e9 / peak, 4)},
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        g, passes, el, cores, g1 = parallel_oracle(args.config, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(g, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                "one_core_value": round(g1, 4),
                                "sample": f"whole batch of {args.config}, {passes} pass(es) in {el:.1f} s "
                                          f"on {cores} worker processes (sequences interleaved); "
                                          f"one core: whole batch on one worker"}
    # the other workloads (one GPU, default configuration only)
    if world == 1 and not args.no_per_config and args.config == DEFAULT_CONFIG and w == W.get(args.config):
        del scn, g_steps, g_attns, g_step, g_attn
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        per = {}
        for cfg in OTHER_CONFIGS:
            e = per_config_entry(cfg, args, dev_name, local, peak)
            if not args.no_cpu_baseline:
                e["cpu_baseline"] = oracle_sample(cfg, args.per_config_cpu_seconds)
            per[cfg] = e
        line["per_config"] = per
    if rank == 0:
        print(json.dumps(line), flush=True)


class CudaRuntime:
    """The CUDA runtime's asynchronous copy and event calls through ctypes, for
    the end-to-end loop: each is one C call, where torch's stream context,
    copy and event wrappers cost several microseconds of host time apiece,
    which a host-bound loop pays every step.  The runtime is the one this
    process already mapped (torch's), else the toolkit's."""

    H2D, D2H = 1, 2

    def __init__(self):
        import ctypes
        paths = []
        try:
            with open("/proc/self/maps") as f:
                for line in f:
                    path = line.split()[-1] if "/" in line else ""
                    if os.path.basename(path).startswith("libcudart") and path not in paths:
                        paths.append(path)
        except OSError:
            pass
        paths += ["/usr/local/cuda/lib64/libcudart.so", "libcudart.so"]
        self.rt = None
        for p in paths:
            try:
                self.rt = ctypes.CDLL(p)
                break
            except OSError:
                continue
        if self.rt is None:
            raise OSError("no CUDA runtime library found")
        vp, c = ctypes.c_void_p, ctypes
        self.rt.cudaMemcpyAsync.argtypes = [vp, vp, c.c_size_t, c.c_int, vp]
        self.rt.cudaEventCreateWithFlags.argtypes = [c.POINTER(vp), c.c_uint]
        self.rt.cudaEventRecord.argtypes = [vp, vp]
        self.rt.cudaStreamWaitEvent.argtypes = [vp, vp, c.c_uint]
        self.rt.cudaEventSynchronize.argtypes = [vp]
        self.rt.cudaEventDestroy.argtypes = [vp]
        self.events = []

    def event(self):
        import ctypes
        e = ctypes.c_void_p()
        if self.rt.cudaEventCreateWithFlags(ctypes.byref(e), 2) != 0:  # timing disabled
            raise RuntimeError("cudaEventCreateWithFlags failed")
        self.events.append(e)
        return e

    def close(self):
        for e in self.events:
            self.rt.cudaEventDestroy(e)
        self.events = []


def end_to_end(scn, dev_name, n: int, world: int, kv_bytes: int):
    """The step through the C ABI with its inputs copied from pinned host
    memory and its output copied back, every step.  Two input/output buffer
    pairs alternate: step i's host-to-device copy runs on an input-copy
    stream while step i - 1 computes, step i - 1's device-to-host copy on an
    output-copy stream while step i computes, and the host waits for step
    i - 1's output before issuing step i + 1 (one step in flight), as a
    serving loop that overlaps transfers with compute does.  (With one copy
    stream for both directions, step i's input copy would queue behind step
    i - 1's output copy, which waits for step i - 1's compute: no overlap.)
    The step is the library's Prepared calls (arguments checked once, as a
    serving loop re-issuing one step on the same buffers does), and the copies
    and events go to the CUDA runtime directly; the loop is host-bound
    otherwise.  Inputs per step: q, the new K/V, block tables and context
    lengths packed in one pinned buffer (one copy); output: the attention
    result.  GB/s over the host's wall clock.  The graph figure (copy in,
    step, copy out captured as one CUDA graph, one replay and one host sync
    per step) is reported beside it."""
    import copy as _copy
    import torch
    names = ("q", "k_new", "v_new", "tables", "ctx")
    slots = []
    for _ in range(2):
        dev_in, views = packed([getattr(scn, n) for n in names], dev_name)
        s = _copy.copy(scn)
        for n_, v_ in zip(names, views):
            setattr(s, n_, v_)
        s.out = torch.empty_like(scn.out)
        host_in = dev_in.cpu().pin_memory()
        host_out = torch.empty_like(scn.out, device="cpu").pin_memory()
        slots.append({"scn": s, "dev_in": dev_in, "host_in": host_in, "host_out": host_out,
                      "step": s.prepare_step()})
    h2d = slots[0]["host_in"].numel()
    d2h = slots[0]["host_out"].numel() * slots[0]["host_out"].element_size()
    compute = torch.cuda.current_stream()
    in_s = torch.cuda.Stream(device=dev_name)
    out_s = torch.cuda.Stream(device=dev_name)
    try:
        rt = CudaRuntime()
        for sl in slots:
            sl["in_ev"], sl["done_ev"], sl["out_ev"] = rt.event(), rt.event(), rt.event()
            sl["p"] = (sl["dev_in"].data_ptr(), sl["host_in"].data_ptr(), sl["scn"].out.data_ptr(),
                       sl["host_out"].data_ptr())
        hc, hi, ho = compute.cuda_stream, in_s.cuda_stream, out_s.cuda_stream

        def issue(i):
            # step i - 2 used this pair: the host has already waited for its output
            sl = slots[i % 2]
            di, hin, do, hout = sl["p"]
            r = rt.rt
            r.cudaMemcpyAsync(di, hin, h2d, rt.H2D, hi)
            r.cudaEventRecord(sl["in_ev"], hi)
            r.cudaStreamWaitEvent(hc, sl["in_ev"], 0)
            sl["step"](hc)
            r.cudaEventRecord(sl["done_ev"], hc)
            r.cudaStreamWaitEvent(ho, sl["done_ev"], 0)
            r.cudaMemcpyAsync(hout, do, d2h, rt.D2H, ho)
            r.cudaEventRecord(sl["out_ev"], ho)

        def wait_out(i):
            if rt.rt.cudaEventSynchronize(slots[i % 2]["out_ev"]) != 0:
                raise RuntimeError("cudaEventSynchronize failed")
        how = "CUDA runtime calls through ctypes"
    except (OSError, RuntimeError, AttributeError):
        rt = None
        for sl in slots:
            sl["in_ev"], sl["done_ev"], sl["out_ev"] = (torch.cuda.Event(), torch.cuda.Event(),
                                                        torch.cuda.Event())

        def issue(i):
            sl = slots[i % 2]
            with torch.cuda.stream(in_s):
                sl["dev_in"].copy_(sl["host_in"], non_blocking=True)
            sl["in_ev"].record(in_s)
            compute.wait_event(sl["in_ev"])
            sl["step"](compute)
            sl["done_ev"].record(compute)
            out_s.wait_event(sl["done_ev"])
            with torch.cuda.stream(out_s):
                sl["host_out"].copy_(sl["scn"].out, non_blocking=True)
            sl["out_ev"].record(out_s)

        def wait_out(i):
            slots[i % 2]["out_ev"].synchronize()
        how = "torch copies and events"

    def run(n):
        for i in range(n):
            issue(i)
            if i >= 1:
                wait_out(i - 1)   # step i - 1's output is on the host
        wait_out(n - 1)

    run(4)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    run(n)
    e2e_s = max_over_ranks((time.perf_counter() - t0) / n, world)
    torch.cuda.synchronize()
    if rt is not None:
        rt.close()
    e2e = {"value": round(world * kv_bytes / e2e_s / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_s * 1e3, 4), "steps": n,
           "what": "host-to-device copy of the step's inputs and device-to-host copy of its output "
                   "every step, two buffer pairs alternating so that copies overlap the previous "
                   "step's compute; the step as the library's prepared calls; copies and events "
                   "by " + how + "; host wall clock"}
    g = None
    if world == 1:
        s0 = slots[0]

        def serial_step():
            s0["dev_in"].copy_(s0["host_in"], non_blocking=True)
            s0["scn"].step()
            s0["host_out"].copy_(s0["scn"].out, non_blocking=True)
            torch.cuda.synchronize()
        g = e2e_graph_of(serial_step, s0["dev_in"], s0["host_in"], s0["scn"], s0["host_out"], n, kv_bytes)
    return e2e, g


# ------------------------------------------------------------------ prefill
PREFILL_METRIC = "paged prefill attention TFLOP/s (causal, algorithmic) & fraction of GB300 bf16 tensor peak"


def prefill_flops(w, ctx, n) -> int:
    """Algorithmic FLOPs of causal chunked prefill: each query at position p
    multiplies with p + 1 keys and values, 4 D flops per (query head, key)."""
    return int(sum(4 * w.head_dim * w.num_q_heads * (int(n[i]) * (int(ctx[i]) - int(n[i])) +
                                                     int(n[i]) * (int(n[i]) + 1) // 2)
                   for i in range(len(ctx))))


class PrefillOracle:
    """The CPU oracle's prefill attention over a bounded sample of sequences
    of the workload (the pool built once, not timed)."""

    def __init__(self, config: str, n_seqs: int = 2):
        import numpy as np
        import workloads as W
        from oracle import scenario as OS
        self.w = w = W.get(config)
        self.scn = OS.build(w, write_seqs=list(range(n_seqs)))
        self.rows = list(range(n_seqs))
        ctx = self.scn.ctx
        self.n = W.chunk_lens(w, ctx, w.prefill_chunk)
        self.qs = np.concatenate([[0], np.cumsum(self.n)])
        self.q = np.concatenate([W.q_for_chunk(w, s, int(self.n[r])).double().numpy()
                                 for r, s in enumerate(self.scn.seq_ids)])
        self.flops = prefill_flops(w, ctx[:n_seqs], self.n[:n_seqs])

    def one_pass(self) -> float:
        import math
        from oracle import prefill as OP
        t0 = time.perf_counter()
        OP.paged_attention_prefill(self.q, self.scn.pool, self.scn.tables, self.scn.ctx, self.qs,
                                   1.0 / math.sqrt(self.w.head_dim), seqs=self.rows)
        return time.perf_counter() - t0


def run_prefill_reference(args, world, rank):
    if rank != 0:
        return
    r = OraclePool(args.config)
    try:
        for _ in range(args.warmup):
            r.one_pass()
        t = [r.one_pass() for _ in range(args.steps)]
    finally:
        r.close()
    sec = statistics.mean(t)
    tf = r.flops / sec / 1e12
    sample = f"whole batch of {args.config}, one pass per step on {r.n} worker processes"
    line = {"metric": PREFILL_METRIC, "value": round(tf, 6), "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": args.config, "flops_per_step": r.flops},
            "cpu_baseline": {"value": round(tf, 6), "unit": "TFLOP/s", "cores": r.n, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(tf, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_prefill_gpu(args, world, rank, local):
    import math
    import numpy as np
    import torch
    import workloads as W
    import paged_kv_cache_137_gb300 as pkv
    from paged_kv_cache_137_gb300 import scenario as PS

    pkv.build()
    torch.cuda.set_device(local)
    dev_name = f"cuda:{local}"
    w = workload_of(args)
    sc = {}
    if w.kv_dtype == "e4m3":
        sc = W.fp8_head_scales(w) if args.fp8_scales == "head" else W.fp8_scales(*W.kv_amax(w))
    scn = PS.materialize(PS.plan(w), dev_name, sc)
    scn.copy_blocks()
    scn.write_step()
    ctx = scn.plan.ctx
    n = W.chunk_lens(w, ctx, w.prefill_chunk)
    qs_np = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    total_q = int(qs_np[-1])
    q = torch.cat([W.q_for_chunk(w, s, int(n[r])) for r, s in enumerate(scn.plan.seq_ids)])
    out = torch.empty_like(q, device=dev_name)
    qs = torch.from_numpy(qs_np).to(dev_name)
    # the chunk's K/V and slots (the same values the pool already holds)
    kv = [W.kv_for_seq(w, s, int(n[r]), first_pos=int(ctx[r]) - int(n[r]))
          for r, s in enumerate(scn.plan.seq_ids)]
    k_new = torch.cat([k for k, _ in kv])
    v_new = torch.cat([v for _, v in kv])
    slots_np = np.concatenate([
        [int(scn.plan.tables[r][p // w.block_size]) * w.block_size + p % w.block_size
         for p in range(int(ctx[r]) - int(n[r]), int(ctx[r]))] for r in range(len(ctx))]).astype(np.int64)
    slots = torch.from_numpy(slots_np)
    # the step's inputs in one device buffer (one host-to-device copy end to end)
    dev_in, (q, k_new, v_new, slots) = packed([q, k_new, v_new, slots], dev_name)
    scale = 1.0 / math.sqrt(w.head_dim)
    max_q = int(n.max())
    flops = prefill_flops(w, ctx, n)
    stream = torch.cuda.current_stream()

    ks, vs = scn.scales.get("k_scale", 1.0), scn.scales.get("v_scale", 1.0)

    def attend():
        pkv.pkv_attention_prefill(out, q, scn.k_cache, scn.v_cache, scn.tables, scn.ctx, qs, scn.desc,
                                  scale, max_query_len=max_q, k_scale=ks, v_scale=vs)

    kinv, vinv = scn.scales.get("k_inv_scale", 1.0), scn.scales.get("v_inv_scale", 1.0)

    def step():
        pkv.pkv_write(scn.k_cache, scn.v_cache, k_new, v_new, slots, scn.desc, kinv, vinv)
        attend()

    side = torch.cuda.Stream(device=dev_name)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for _ in range(max(args.warmup, 3)):
            step()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    # the K steps (and K attention calls) captured back to back in one graph,
    # each graph replayed back to back for at least --timed-ms of device time
    K = args.steps
    g_steps, g_attns = capture(step, K), capture(attend, K)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        step_reps = replay_timed(g_steps, stream, args.timed_ms)
        torch.cuda.synchronize()
        barrier(world)
        attn_reps = replay_timed(g_attns, stream, args.timed_ms / 2)
    ms = max_over_ranks(statistics.median(step_reps) / K, world)
    attn = statistics.median(attn_reps) / K
    value = world * flops / (ms / 1e3) / 1e12

    # end to end through the C ABI from pinned host buffers: q, the chunk's
    # K/V and slots packed in one pinned buffer and copied in once, the
    # output copied back, then a sync
    host_in = dev_in.cpu().pin_memory()
    out_host = torch.empty_like(out, device="cpu").pin_memory()
    h2d = host_in.numel()
    d2h = out_host.numel() * out_host.element_size()

    def e2e_step():
        dev_in.copy_(host_in, non_blocking=True)
        step()
        out_host.copy_(out, non_blocking=True)
        torch.cuda.synchronize()

    for _ in range(3):
        e2e_step()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(min(K, 50)):
        e2e_step()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / min(K, 50), world)

    d = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak, peak_kind = (float(d["bf16_tflops"]), "measured") if "bf16_tflops" in d else (1900.0, "fallback")
    peak_sustained = float(d.get("bf16_tflops_sustained", 1700.0))
    achieved = flops / (attn / 1e3) / 1e12
    # the step's inputs: queries and the K/V of the chunks' contexts
    in_bytes = (total_q * w.num_q_heads * w.head_dim * 2
                + 2 * int(ctx.sum()) * w.num_kv_heads * w.head_dim * w.kv_bytes)
    l2_bytes = torch.cuda.get_device_properties(local).L2_cache_size
    pf_kernel = ("prefill_umma_kernel (tcgen05.mma, TMEM accumulators)"
                 if w.head_dim == 128
                 else "prefill_tc_kernel (mma.sync m16n8k16)")
    line = {
        "metric": PREFILL_METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": K, "warmup": max(args.warmup, 3), "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.kv_dtype,
        "data": "synthetic",
        "config": {"workload": args.config, "num_seqs": w.num_seqs, "num_q_heads": w.num_q_heads,
                   "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
                   "chunk": w.prefill_chunk, "query_tokens": total_q, "kv_dtype": w.kv_dtype,
                   **({"fp8_scales": args.fp8_scales} if w.kv_dtype == "e4m3" else {}),
                   "context_tokens": int(ctx.sum()), "flops_per_step": flops,
                   "l2": ("inputs %s than L2 (q + K/V %d MB vs %d MB L2), no flush between steps"
                          % ("larger" if in_bytes > l2_bytes else "smaller", in_bytes >> 20,
                             l2_bytes >> 20)),
                   "launch": ("the K steps captured back to back in one CUDA graph; the graph replayed "
                              "%d times back to back (%.0f ms timed), median replay / K"
                              % (len(step_reps), sum(step_reps))),
                   "parallelism": "replicas" if world > 1 else "single"},
        "tokens_per_s": round(world * total_q / (ms / 1e3), 1),
        "roofline": {"bound": "tensor", "kernel": pf_kernel,
                     "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} bf16 burst",
                     "peak_sustained": peak_sustained,
                     "frac_of_sustained": round(achieved / peak_sustained, 4),
                     "traffic": traffic_for(args.config, pf_kernel) if w == W.get(args.config) else None,
                     "attention_ms": round(attn, 4)},
        "e2e": {"value": round(world * flops / e2e_s / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_s * 1e3, 4)},
        "gpu_launches": 2 * K * (len(step_reps) + 1) + K * (len(attn_reps) + 1),
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        g, passes, el, cores, g1 = parallel_oracle(args.config, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(g, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "one_core_value": round(g1, 6),
                                "sample": f"whole batch of {args.config}, {passes} pass(es) in {el:.1f} s "
                                          f"on {cores} worker processes (sequences interleaved); "
                                          f"one core: whole batch on one worker"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    # the oracle is timed on one host thread
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ.setdefault(v, "1")
    world, rank, local = dist_setup(args)
    import workloads as W
    prefill = W.get(args.config).prefill_chunk > 0
    if args.impl == "reference":
        (run_prefill_reference if prefill else run_reference)(args, world, rank)
    else:
        (run_prefill_gpu if prefill else run_gpu)(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
