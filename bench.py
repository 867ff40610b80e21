"""Benchmark: one paged-attention decode step of the Llama-2-7B-shaped layer.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 7b] [--impl reference]

A step = swap_out -> swap_in -> copy_blocks -> reshape_and_cache -> paged decode
(+ log-sum-exp merge) for one layer of the workload (the 7B workload has no
swaps or copies).  The KV pool (2.9 GB, > L2) stays resident; per-step inputs are
already in HBM when the timed region starts.  Prints one JSON line.

value  = algorithmic bytes of the step / device time of the step, GB/s (whole job).
e2e    = the same, through the C ABI with host buffers: every step copies the
         step's inputs (q, new K/V, block tables, context lengths, slot mapping)
         from one pinned host buffer and the output back, inside the timed region.
roofline = the decode launch (pa_decode: decode kernel + merge kernel) against the
         measured HBM copy bandwidth.
--impl reference times the fp64 CPU oracle (the correctness reference) on a
bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "paged-attn decode KV-read HBM GB/s (frac of peak); seq-steps/s at 7B shape"
SPEC_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
DESCRIPTIONS = {
    "tiny": "tiny paged decode: 4 seqs, MHA 4 heads, head_size 64, block_size 16, fp16, ctx U[1,100]",
    "7b": "Llama-2-7B-shaped decode layer: 64 seqs, 32 q/32 kv heads, head_size 128, block_size 16, fp16 "
          "K/V/Q ~N(0,1), context_lens ~U[512,4096], pool 1.2x needed blocks, random block_tables, "
          "reshape_and_cache of 1 token/seq",
    "8b": "Llama-3-8B-shaped GQA decode: 256 seqs, 32 q/8 kv heads, head_size 128, block_size 16, bf16, "
          "context_lens lognormal(median 1024, sigma 0.8) capped at 8192",
    "70b": "long-context 70B-shaped GQA decode: 8 seqs, 64 q/8 kv heads, head_size 128, block_size 32, bf16, "
           "context_lens ~U[32768,131072]",
    "beam": "beam/shared-prefix decode: 32 groups x 4 beams, 32 q/8 kv heads, head_size 128, block_size 16, "
            "bf16, 2048-token shared prompt, tails ~U[0,256], CoW copy_blocks + 10% swap_blocks",
    "7b_bs1": "Llama-2-7B-shaped decode layer with token-granular paging (block_size 1): 64 seqs, 32/32 heads, "
              "head_size 128, fp16, context_lens ~U[512,4096]",
    "7b_int8": "Llama-2-7B-shaped decode layer over an 8-bit KV cache (int8 codes + fp32 scale per token and "
               "kv head): 64 seqs, 32/32 heads, head_size 128, block_size 16, fp16 q/out, history K/V ~N(0,1) "
               "quantised by the library's writer, context_lens ~U[512,4096]",
    "8b_int8": "Llama-3-8B-shaped GQA decode over an 8-bit KV cache: 256 seqs, 32 q/8 kv heads, head_size 128, "
               "block_size 16, bf16 q/out, context_lens lognormal(median 1024, sigma 0.8) capped at 8192",
}


PREFILL_METRIC = "paged prefill/extend attention TFLOP/s (causal FLOPs, frac of bf16 tensor peak)"
FALLBACK_BF16_TFLOPS = 1900.0
PREFILL_DESCRIPTIONS = {
    "prefill_8b": "Llama-3-8B-shaped prefill: 16 prompts x 2048 tokens from scratch, 32 q/8 kv heads, head_size 128, "
                  "block_size 16, bf16 ~N(0,1), random block placement; reshape_and_cache of every prompt token + "
                  "causal paged attention",
    "extend_8b": "Llama-3-8B-shaped chunked prefill: 32 sequences, a 512-token chunk each over cached prefixes "
                 "~U[512,3584], 32 q/8 kv heads, head_size 128, block_size 16, bf16",
    "prefill_7b": "Llama-2-7B-shaped prefill: 8 prompts x 2048 tokens, 32/32 heads, head_size 128, block_size 16, fp16",
    "prefill_tiny": "tiny prefill: 3 sequences, 100-token chunks over prefixes ~U[0,300], 8 q/2 kv heads, bf16",
}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    """bf16 dense TFLOP/s: burst figure (a kernel timed alone)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (burst)"
    return FALLBACK_BF16_TFLOPS, "fallback"


# the sources the decode launch (tensor-core decode + log-sum-exp merge) is built from
DECODE_SOURCES = ("common.cuh", "tc_common.cuh", "kernels.h", "decode_tc.cuh", "decode_tc.cu", "decode_tc_prefix.cu",
                  "decode_simt.cu")


def source_digest() -> str:
    """Digest of the decode kernels' sources: a recorded DRAM-traffic figure is used
    only while it was taken on these exact sources."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_168_gb300", "csrc")
    for name in DECODE_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, partition_size: int):
    """DRAM bytes per decode launch from the committed ncu summary, if it was taken
    on the current kernel sources at this partition size (else None)."""
    path = os.path.join(ROOT, "profiles", f"decode_{workload}_traffic.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_src = re.search(r"source_digest:\s*([0-9a-f]+)", text)
    m_val = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_part = re.search(r"partition_size:\s*([0-9]+)", text)
    if not (m_src and m_val and m_part) or m_src.group(1) != source_digest() or int(m_part.group(1)) != partition_size:
        return None
    return float(m_val.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background; only samples taken
    inside the timed window (mark_start / mark_end, host clock) are summarised."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int, interval_ms: int = 50):
        self.index, self.interval_ms, self.proc, self.lines = index, interval_ms, None, []
        self.t0 = self.t1 = self.tt = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms",
                 str(self.interval_ms), "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_timed(self):
        self.tt = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    @staticmethod
    def _parse(line):
        import datetime
        f = [x.strip() for x in line.split(",")]
        if len(f) < 10:
            return None
        try:
            ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            return ts, float(f[2]), float(f[3]), f[6:10]
        except ValueError:
            return None

    def summary(self, soak_steps: int = 0):
        """Median SM clock and throttle reasons over the samples taken between
        mark_start and mark_end (the pre-timing soak and the timed steps)."""
        samples = [x for x in (self._parse(ln) for ln in self.lines) if x]
        if not samples:
            return None
        inside = [x for x in samples if self.t0 is not None and self.t0 <= x[0] <= (self.t1 or x[0])]
        timed = [x for x in inside if self.tt is None or x[0] >= self.tt]
        used = inside or [min(samples, key=lambda x: abs(x[0] - (self.t0 or x[0])))]
        reasons = sorted({name for x in used for name, v in zip(self.REASONS, x[3]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median([x[1] for x in used])), "sm_max_mhz": max(x[2] for x in used),
                "reasons": reasons, "samples": len(used), "samples_in_timed_region": len(timed),
                "window": f"{soak_steps} untimed steps right before the timed ones, then the timed steps"}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(x: float, world: int, device) -> float:
    """Max over ranks (identity on one process)."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class HostInputs:
    """A step's inputs packed into one pinned host buffer, so each end-to-end step
    moves them with one host->device copy (small copies each pay the link's
    latency); on the device each input is a view of one staging buffer, every
    view 256-byte aligned."""

    def __init__(self, w, names, device):
        offs, at = {}, 0
        for k in names:
            t = getattr(w, k)
            offs[k] = at
            at += -(-t.numel() * t.element_size() // 256) * 256
        self.host = torch.zeros(at, dtype=torch.uint8).pin_memory()
        self.dev = torch.empty(at, dtype=torch.uint8, device=device)
        self.views = {}
        for k in names:
            t = getattr(w, k).contiguous()
            n = t.numel() * t.element_size()
            self.host[offs[k]:offs[k] + n].copy_(t.reshape(-1).view(torch.uint8).cpu())
            self.views[k] = self.dev[offs[k]:offs[k] + n].view(t.dtype).view(t.shape)
        self.nbytes = at

    def upload(self):
        self.dev.copy_(self.host, non_blocking=True)


def decode_config(w, args, world: int) -> dict:
    """The `config` object of a decode line, identical in both arms: the workload,
    its batch and context sizes, the partition size pa_decode takes for it, the
    parallelism, and how the step compares with the L2."""
    from paged_kv_cache_168_gb300 import _lib
    cfg = w.cfg
    desc = _lib.CacheDesc(w.num_blocks, cfg.block_size, cfg.num_kv_heads, cfg.head_size, w.dtype,
                          kv_int8=cfg.kv_int8)
    if w.group_start is not None:      # shared prompt blocks: pa_decode_shared_prefix's partition
        part = _lib.decode_shared_prefix_partition_size(desc, cfg.num_seqs, cfg.num_q_heads, len(w.prefix_lens_np),
                                                        w.max_context_len, args.partition_size)
    else:
        part = _lib.decode_partition_size(desc, cfg.num_seqs, w.max_context_len, args.partition_size)
    ctx = w.context_lens_np.astype(np.int64)
    kv_tok = cfg.num_kv_heads * (2 * cfg.head_size + 8) if cfg.kv_int8 else 2 * cfg.num_kv_heads * cfg.head_size * 2
    return {"workload": DESCRIPTIONS[args.workload] + (f" (first {args.seqs} sequences)" if args.seqs else ""),
            "global_batch": cfg.num_seqs * world, "max_context_len": w.max_context_len,
            "tokens_in_context": int(ctx.sum()), "partition_size": part, "parallelism": f"replicas{world}",
            "l2": f"inputs larger than L2: {_lib.cache_bytes(desc) / 1e9:.2f} GB pool, "
                  f"{int(ctx.sum()) * kv_tok / 1e9:.2f} GB of KV read per step"}


# ------------------------------------------------------------------ CPU oracle timing

_ORACLE_INPUTS = {}


def oracle_inputs(w):
    """Host copies (raw 16-bit bits) of the workload for the oracle, made once.
    An 8-bit cache starts as an empty oracle pool that oracle_build_blocks fills."""
    import oracle
    from paged_kv_cache_168_gb300.workloads import as_u16
    key = id(w)
    if key not in _ORACLE_INPUTS:
        cfg = w.cfg
        g = oracle.Geom(w.num_blocks, cfg.block_size, cfg.num_kv_heads, cfg.head_size, cfg.dtype)
        if cfg.kv_int8:
            pool = np.zeros(w.num_blocks * oracle.i8_block_bytes(g), np.uint8)
            built = np.zeros(w.num_blocks, dtype=bool)
            _ORACLE_INPUTS[key] = (g, pool, as_u16(w.q), built)
        else:
            _ORACLE_INPUTS[key] = (g, as_u16(w.kv_cache).reshape(-1), as_u16(w.q), None)
    return _ORACLE_INPUTS[key]


def oracle_build_blocks(w, s):
    """8-bit cache: the oracle quantises sequence s's blocks from the workload's
    logical history (blocks it has not built yet)."""
    import oracle
    from paged_kv_cache_168_gb300.workloads import as_u16
    g, pool, _, built = oracle_inputs(w)
    bs = w.cfg.block_size
    blocks = w.block_tables_np[s, :-(-int(w.context_lens_np[s]) // bs)]
    blocks = np.unique(blocks[~built[blocks]])
    if blocks.size == 0:
        return
    part = w.kv_logical[torch.from_numpy(blocks).to(w.kv_logical.device)]        # [n, Hkv, 2, bs, D]
    n, hkv, _, _, d = part.shape
    key = as_u16(part[:, :, 0].permute(0, 2, 1, 3).reshape(n * bs, hkv, d))
    value = as_u16(part[:, :, 1].permute(0, 2, 1, 3).reshape(n * bs, hkv, d))
    slots = (blocks[:, None].astype(np.int64) * bs + np.arange(bs)).reshape(-1)
    assert oracle.reshape_and_cache_i8(pool, g, key, value, slots) == 0
    built[blocks] = True


def oracle_sample(w, budget_s: float, max_items: int | None = None, start: int = 0, threads: int = 0):
    """Time the fp64 oracle on the workload sequence by sequence (all query heads
    of a sequence together) until ~budget_s seconds of wall time, on `threads`
    OpenMP threads (0: all).  Returns (GB/s of algorithmic KV bytes, seq-steps/s,
    description, cores, seconds)."""
    import oracle
    cfg = w.cfg
    g, pool, q, _ = oracle_inputs(w)
    kv_tok = cfg.num_kv_heads * (2 * cfg.head_size + 8) if cfg.kv_int8 else 2 * cfg.num_kv_heads * cfg.head_size * 2
    done_bytes, done_seqs, t_total = 0, 0, 0.0
    order = np.random.default_rng(start).permutation(cfg.num_seqs)
    for s in order:
        if cfg.kv_int8:
            oracle_build_blocks(w, s)           # cache construction, not timed
            t0 = time.perf_counter()
            oracle.decode_i8(q[s:s + 1], pool, g, w.block_tables_np[s:s + 1], w.context_lens_np[s:s + 1],
                             w.scale, max_context_len=w.max_context_len, nthreads=threads)
        else:
            sel = np.array([[s, h] for h in range(cfg.num_q_heads)], dtype=np.int32)
            t0 = time.perf_counter()
            oracle.decode(q, pool, g, w.block_tables_np, w.context_lens_np, w.scale,
                          max_context_len=w.max_context_len, sel=sel, nthreads=threads)
        t_total += time.perf_counter() - t0
        done_bytes += int(w.context_lens_np[s]) * kv_tok
        done_seqs += 1
        if t_total >= budget_s or (max_items and done_seqs >= max_items):
            break
    cores = threads or oracle.max_threads()
    desc = (f"{done_seqs} of {cfg.num_seqs} sequences (all {cfg.num_q_heads} query heads each, "
            f"{done_bytes / 1e9:.3f} GB of KV) of the {cfg.name} workload, fp64 oracle, {cores} OpenMP threads")
    return done_bytes / t_total / 1e9, done_seqs / t_total, desc, cores, t_total


def run_reference_prefill(args):
    """The fp64 oracle's prefill on the host cores, on windows of the prefill workload."""
    from paged_kv_cache_168_gb300.workloads import make_prefill_workload
    w = make_prefill_workload(args.workload, device="cpu")
    cfg = w.cfg
    per_step = max(1.0, args.reference_seconds / max(args.steps + args.warmup, 1))
    for i in range(args.warmup):
        prefill_oracle_sample(w, per_step / 4, start=100 + i)
    vals, desc, cores = [], "", 1
    for i in range(args.steps):
        v, desc, cores = prefill_oracle_sample(w, per_step, start=i + 1)
        vals.append(v)
    value = float(np.median(vals))
    line = {
        "impl": "reference", "metric": PREFILL_METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * per_step, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": PREFILL_DESCRIPTIONS[args.workload], "global_batch": cfg.num_seqs},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": "each step: " + desc},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference(args):
    world, rank, local = dist_env()
    if rank != 0:
        return 0
    if args.workload in PREFILL_DESCRIPTIONS:
        return run_reference_prefill(args)
    from paged_kv_cache_168_gb300.build import build
    from paged_kv_cache_168_gb300.workloads import make_workload
    build()                                   # host-side sizes (the partition size in `config`)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = make_workload(args.workload, device=dev, num_seqs=args.seqs)
    cfg = w.cfg
    # each step is a bounded sample: a few sequences of the workload
    per_step = max(1.0, args.reference_seconds / max(args.steps + args.warmup, 1))
    for _ in range(args.warmup):
        oracle_sample(w, per_step / 4, max_items=1)
    vals, seqs, secs, desc, cores = [], [], [], "", 1
    for i in range(args.steps):
        v, sps, desc, cores, t = oracle_sample(w, per_step, start=i + 1)
        vals.append(v)
        seqs.append(sps)
        secs.append(t)
    value = float(np.median(vals))
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * float(np.median(secs)), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": decode_config(w, args, world),
        "seq_steps_per_s": round(float(np.median(seqs)), 4),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": "each step: " + desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU benchmark

def run_gpu(args):
    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        print(json.dumps({"metric": METRIC, "error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    from paged_kv_cache_168_gb300 import _lib
    from paged_kv_cache_168_gb300.build import build
    from paged_kv_cache_168_gb300.step import DecodeStep
    from paged_kv_cache_168_gb300.workloads import CONFIGS, make_workload
    build()
    _lib.load()

    cfg = CONFIGS[args.workload]
    w = make_workload(args.workload, device=device, seed=cfg.seed + 1000 * rank, num_seqs=args.seqs)
    stream = torch.cuda.Stream(device)
    step = DecodeStep(w, partition_size=args.partition_size, stream=stream, nvtx=True)
    nbytes = step.algorithmic_bytes()
    torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    check_device_errors(_lib, step, stream, "warm-up")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        # the clock record covers the timed steps and, right before them, the same
        # step repeated for ~soak seconds (untimed): a timed region of a few ms is
        # shorter than nvidia-smi's sampling interval
        clocks.mark_start()
        soak_steps = soak(step, stream, args.clock_soak_seconds)
        torch.cuda.synchronize()
        clocks.mark_timed()
        with torch.cuda.stream(stream):
            for i in range(K):
                ev[i][0].record(stream)
                step.cache_ops()
                ev[i][1].record(stream)
                step.attention()
                ev[i][2].record(stream)
                ev[i][3].record(stream)
        torch.cuda.synchronize()
        clocks.mark_end()
        barrier(world)
    total_ms = ev[0][0].elapsed_time(ev[K - 1][3])
    decode_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    total_ms = reduce_max(total_ms, world, device)
    check_device_errors(_lib, step, stream, "the soak and timed steps")

    # ---- end to end through the C ABI with host buffers
    names = ("q", "key", "value", "block_tables", "context_lens", "slot_mapping")
    staged = HostInputs(w, names, device)
    host_out = torch.empty(w.q.shape, dtype=w.q.dtype).pin_memory()
    h2d = staged.nbytes
    d2h = host_out.numel() * host_out.element_size()
    saved = {k: getattr(w, k) for k in names}
    for k in names:
        setattr(w, k, staged.views[k])

    def e2e_step():
        staged.upload()
        step()
        host_out.copy_(step.out, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup)):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            e2e_step()
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = reduce_max(e0.elapsed_time(e1), world, device)
    for k, v in saved.items():
        setattr(w, k, v)

    ms = total_ms / K
    value = world * nbytes["total"] / (ms * 1e-3) / 1e9
    dec_ms = float(np.mean(decode_ms))
    achieved = nbytes["decode_unique"] / (dec_ms * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    part = step.partition()
    step_sp = step.shared_prefix
    launches = K * step.kernel_launches() * world
    del step
    extras = {}
    for name in [x for x in args.extra_workloads.split(",") if x and x != args.workload]:
        extras[name] = measure_workload(name, args, device, stream, peak, rank)

    line = None
    if rank == 0:
        cpu = None
        if args.cpu_baseline_seconds > 0:
            v, sps, desc, cores, _ = oracle_sample(w, args.cpu_baseline_seconds)
            v1, sps1, desc1, _, _ = oracle_sample(w, args.cpu_baseline_seconds / 3, start=7, threads=1)
            cpu = {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc,
                   "seq_steps_per_s": round(sps, 4),
                   "single_thread": {"value": round(v1, 4), "unit": "GB/s", "cores": 1, "sample": desc1,
                                     "seq_steps_per_s": round(sps1, 4)}}
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.cfg.dtype + ("+int8 cache" if w.cfg.kv_int8 else ""),
            "data": "synthetic",
            "config": decode_config(w, args, world),
            "seq_steps_per_s": round(world * w.cfg.num_seqs / (ms * 1e-3), 1),
            "decode_kv_gbs": round(nbytes["decode_kv"] / (dec_ms * 1e-3) / 1e9, 2),
            "decode_unique_kv_gbs": round(nbytes["decode_kv_unique"] / (dec_ms * 1e-3) / 1e9, 2),
            "decode_ms_p10_p50_p90": [round(float(np.percentile(decode_ms, x)), 4) for x in (10, 50, 90)],
            "frac_of_spec_8tbs": round(achieved / SPEC_HBM_GBS, 4),
            "bytes_per_step": nbytes,
            "roofline": {"bound": "hbm", "kernel": ("pa_decode_shared_prefix" if step_sp else "pa_decode")
                                                   + " (decode + log-sum-exp merge)",
                         "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                         "bytes": "algorithmic decode bytes, a shared physical block's tokens counted once",
                         "traffic": recorded_traffic(args.workload, part),
                         "decode_ms": round(dec_ms, 4)},
            "workloads": extras,
            "cpu_baseline": cpu,
            "e2e": {"value": round(world * nbytes["total"] / (e2e_ms / K * 1e-3) / 1e9, 2), "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": round(e2e_ms / K, 4)},
            "gpu_launches": launches,
            "clocks": clocks.summary(soak_steps),
            "source_digest": source_digest(),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def check_device_errors(_lib, step, stream, where: str) -> None:
    """Fail with the error word's bits (PA_DEVERR_*) if a kernel reported one."""
    bits = _lib.read_device_errors(step.dev_err, stream=stream)
    if bits:
        names = [n for n, b in (("context", _lib.DEVERR_CONTEXT), ("block id", _lib.DEVERR_BLOCK_ID),
                                ("slot", _lib.DEVERR_SLOT), ("timeout", _lib.DEVERR_TIMEOUT),
                                ("prefix", _lib.DEVERR_PREFIX)) if bits & b]
        raise AssertionError(f"device error bits {bits:#x} ({', '.join(names) or 'unknown'}) during {where}")


def soak(step, stream, seconds: float) -> int:
    """Run the step back to back for about `seconds` (untimed); returns the count."""
    if seconds <= 0:
        return 0
    with torch.cuda.stream(stream):
        step()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        step()
        torch.cuda.synchronize()
        per = max(time.perf_counter() - t0, 1e-5)
        n = max(1, int(seconds / per))
        for _ in range(n):
            step()
    return n + 2


def measure_workload(name: str, args, device, stream, peak: float, rank: int) -> dict:
    """Decode of another workload in the same run, under the same warm-up and
    step count as the headline: mean decode time (pa_decode launch), KV GB/s
    (logical and unique bytes) and the roofline fraction on unique bytes.  For a
    workload whose sequences share physical blocks it is also timed with a
    buffer of twice the L2 written between steps, so no step finds the previous
    one's blocks in L2."""
    from paged_kv_cache_168_gb300.step import DecodeStep
    from paged_kv_cache_168_gb300.workloads import CONFIGS, make_workload
    from paged_kv_cache_168_gb300 import _lib
    cfg = CONFIGS[name]
    w = make_workload(name, device=device, seed=cfg.seed + 1000 * rank)
    step = DecodeStep(w, stream=stream, nvtx=True)
    nb = step.algorithmic_bytes()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    K = args.steps

    def timed(flush=None):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
        with torch.cuda.stream(stream):
            for i in range(K):
                if flush is not None:
                    flush.add_(1)
                ev[i][0].record(stream)
                step.cache_ops()
                ev[i][1].record(stream)
                step.attention()
                ev[i][2].record(stream)
        torch.cuda.synchronize()
        return [e[1].elapsed_time(e[2]) for e in ev], [e[0].elapsed_time(e[2]) for e in ev]

    dec, tot = timed()
    check_device_errors(_lib, step, stream, name)
    dec_ms, step_ms = float(np.mean(dec)), float(np.mean(tot))
    uniq = nb["decode_unique"] / (dec_ms * 1e-3) / 1e9
    part = step.partition()
    r = {"workload": DESCRIPTIONS[name], "partition_size": part,
         "call": "pa_decode_shared_prefix" if step.shared_prefix else "pa_decode", "decode_ms": round(dec_ms, 4),
         "decode_ms_p10_p50_p90": [round(float(np.percentile(dec, x)), 4) for x in (10, 50, 90)],
         "decode_kv_gbs": round(nb["decode_kv"] / (dec_ms * 1e-3) / 1e9, 2),
         "decode_unique_kv_gbs": round(nb["decode_kv_unique"] / (dec_ms * 1e-3) / 1e9, 2),
         "roofline": {"bound": "hbm", "achieved": round(uniq, 2), "peak": peak, "unit": "GB/s",
                      "frac": round(uniq / peak, 4), "bytes": "algorithmic decode bytes, shared blocks once",
                      "traffic": recorded_traffic(name, part)},
         "frac_of_spec_8tbs": round(nb["decode_kv_unique"] / (dec_ms * 1e-3) / 1e9 / SPEC_HBM_GBS, 4),
         "seq_steps_per_s": round(cfg.num_seqs / (step_ms * 1e-3), 1),
         "step_ms": round(step_ms, 4), "step_gbs": round(nb["total"] / (step_ms * 1e-3) / 1e9, 2),
         "bytes_per_step": nb, "gpu_launches": K * step.kernel_launches()}
    if nb["decode_kv_unique"] != nb["decode_kv"]:
        props = torch.cuda.get_device_properties(device)
        l2 = int(getattr(props, "L2_cache_size", 0) or 0) or 132 * 1024 * 1024
        flush = torch.zeros(2 * l2 // 4, dtype=torch.int32, device=device)
        dec_f, _ = timed(flush)
        fl_ms = float(np.mean(dec_f))
        r["l2_flushed"] = {"flush_bytes": 2 * l2, "decode_ms": round(fl_ms, 4),
                           "decode_unique_kv_gbs": round(nb["decode_kv_unique"] / (fl_ms * 1e-3) / 1e9, 2),
                           "frac": round(nb["decode_unique"] / (fl_ms * 1e-3) / 1e9 / peak, 4)}
        del flush
    del step, w
    torch.cuda.empty_cache()
    return r


# ------------------------------------------------------------------ prefill / extend

def prefill_oracle_sample(w, budget_s: float, start: int = 0, threads: int = 0):
    """Time the fp64 oracle's prefill on 64-query-token windows of the workload
    (all heads; a window at a random offset of a random sequence, attending
    everything before it) until ~budget_s seconds, on `threads` OpenMP threads
    (0: all): (TFLOP/s of causal FLOPs, description, cores)."""
    import oracle
    from paged_kv_cache_168_gb300.workloads import as_u16
    cfg = w.cfg
    g = oracle.Geom(w.num_blocks, cfg.block_size, cfg.num_kv_heads, cfg.head_size, cfg.dtype)
    pool = as_u16(w.kv_cache).reshape(-1)
    q = as_u16(w.q)
    qsl, ctx = w.query_start_loc_np, w.context_lens_np
    rng = np.random.default_rng(start)
    flops, t_total, windows = 0, 0.0, 0
    while t_total < budget_s and windows < 10000:
        s = int(rng.integers(cfg.num_seqs))
        q_len = int(qsl[s + 1] - qsl[s])
        n = min(q_len, 64)
        j0 = int(rng.integers(0, q_len - n + 1))
        c = int(ctx[s]) - q_len + j0 + n                     # the context the window's last token sees
        t0 = time.perf_counter()
        oracle.prefill(q[qsl[s] + j0:qsl[s] + j0 + n], pool, g, w.block_tables_np[s:s + 1],
                       np.array([c], np.int32), np.array([0, n], np.int32), w.scale, nthreads=threads)
        t_total += time.perf_counter() - t0
        flops += 4 * cfg.head_size * cfg.num_q_heads * (n * (c - n) + n * (n + 1) // 2)
        windows += 1
    cores = threads or oracle.max_threads()
    desc = (f"{windows} windows of 64 query tokens (all {cfg.num_q_heads} heads, random sequence and offset) "
            f"of the {cfg.name} workload, fp64 oracle, {cores} OpenMP threads")
    return flops / t_total / 1e12, desc, cores


def run_gpu_prefill(args):
    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        print(json.dumps({"metric": PREFILL_METRIC, "error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    from paged_kv_cache_168_gb300 import _lib
    from paged_kv_cache_168_gb300.build import build
    from paged_kv_cache_168_gb300.step import PrefillStep
    from paged_kv_cache_168_gb300.workloads import PREFILL_CONFIGS, make_prefill_workload
    build()
    _lib.load()
    cfg = PREFILL_CONFIGS[args.workload]
    w = make_prefill_workload(args.workload, device=device, seed=cfg.seed + 1000 * rank)
    stream = torch.cuda.Stream(device)
    step = PrefillStep(w, stream=stream)
    flops = step.flops()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    check_device_errors(_lib, step, stream, "warm-up")
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        clocks.mark_start()
        with torch.cuda.stream(stream):
            for i in range(K):
                ev[i][0].record(stream)
                step.cache_ops()
                ev[i][1].record(stream)
                step.attention()
                ev[i][2].record(stream)
        torch.cuda.synchronize()
        clocks.mark_end()
        barrier(world)
    total_ms = reduce_max(ev[0][0].elapsed_time(ev[K - 1][2]), world, device)
    attn_ms = float(np.mean([ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]))
    check_device_errors(_lib, step, stream, "the soak and timed steps")

    # end to end with host buffers: inputs in, output back, every step
    names = ("q", "key", "value", "block_tables", "context_lens", "query_start_loc", "slot_mapping")
    staged = HostInputs(w, names, device)
    host_out = torch.empty(w.q.shape, dtype=w.q.dtype).pin_memory()
    h2d = staged.nbytes
    d2h = host_out.numel() * host_out.element_size()
    saved = {k: getattr(w, k) for k in names}
    for k in names:
        setattr(w, k, staged.views[k])

    def e2e_step():
        staged.upload()
        step()
        host_out.copy_(step.out, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup)):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            e2e_step()
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = reduce_max(e0.elapsed_time(e1), world, device)
    for k, v in saved.items():
        setattr(w, k, v)

    ms = total_ms / K
    peak, peak_kind = measured_tensor_peak()
    achieved = flops / (attn_ms * 1e-3) / 1e12
    if rank == 0:
        cpu = None
        if args.cpu_baseline_seconds > 0:
            v, desc, cores = prefill_oracle_sample(w, args.cpu_baseline_seconds)
            v1, desc1, _ = prefill_oracle_sample(w, args.cpu_baseline_seconds / 3, start=7, threads=1)
            cpu = {"value": round(v, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc,
                   "single_thread": {"value": round(v1, 6), "unit": "TFLOP/s", "cores": 1, "sample": desc1}}
        line = {
            "metric": PREFILL_METRIC, "value": round(world * flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype,
            "data": "synthetic",
            "config": {"workload": PREFILL_DESCRIPTIONS[args.workload], "global_batch": cfg.num_seqs * world,
                       "query_tokens": int(w.query_start_loc_np[-1]),
                       "tokens_in_context": int(w.context_lens_np.sum()), "parallelism": f"replicas{world}",
                       "l2": f"inputs larger than L2: q {w.q.numel() * 2 / 1e9:.2f} GB + pool "
                             f"{w.kv_cache.numel() * 2 / 1e9:.2f} GB per step"},
            "flops_per_step": flops,
            "tokens_per_s": round(world * int(w.query_start_loc_np[-1]) / (ms * 1e-3), 1),
            "roofline": {"bound": "tensor", "kernel": "pa_prefill (prefill_tc_kernel)", "achieved": round(achieved, 2),
                         "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                         "traffic": None, "attention_ms": round(attn_ms, 4),
                         "note": "algorithmic causal FLOPs; the kernel also issues the p_lo half of PV and "
                                 "full 128x128 diagonal tiles"},
            "cpu_baseline": cpu,
            "e2e": {"value": round(world * flops / (e2e_ms / K * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms / K, 4)},
            "gpu_launches": K * step.kernel_launches() * world,
            "clocks": clocks.summary(),
            "source_digest": source_digest(),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="7b", choices=sorted(DESCRIPTIONS) + sorted(PREFILL_DESCRIPTIONS))
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--partition-size", type=int, default=0)
    ap.add_argument("--seqs", type=int, default=None, help="use only the first N sequences (small profiling runs)")
    ap.add_argument("--cpu-baseline-seconds", type=float, default=10.0)
    ap.add_argument("--reference-seconds", type=float, default=60.0)
    ap.add_argument("--extra-workloads", default="8b,70b,beam",
                    help="decode workloads also measured in the same run (the line's `workloads`); '' for none")
    ap.add_argument("--clock-soak-seconds", type=float, default=1.0,
                    help="untimed back-to-back steps before the timed ones, inside the clock record")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.workload in PREFILL_DESCRIPTIONS:
        return run_gpu_prefill(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
