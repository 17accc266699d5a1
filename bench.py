"""Benchmark of the paged decode step (KV write + decode attention) at Llama-3-8B GQA shapes.

One step = one layer's pass of the hot path over the serving batch: ``paged_kv_write`` of the 64
new tokens through ``slot_mapping``, then ``paged_attention_decode`` (split-K partitions and the
log-sum-exp merge included) — 32 query / 8 KV heads, head_dim 128, block_size 16, bf16, batch 64,
context lengths uniform in [512, 4096], block tables drawn from a shuffled 40,000-block pool.

Timed on the device with CUDA events after warm-up; steps rotate over several independent layer
pools so that no step finds its K/V in L2 (each step reads ~604 MB; the rotation spans > 2 GB).
Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle instead.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "paged decode attn: KV GB/s (% HBM roofline) and decode tok/s, Llama-3-8B GQA"
UNIT = "GB/s"
HQ, HKV, D, S = 32, 8, 128, 16
SEED_LONG = 1004  # seed of the long-context configuration's device inputs
LLAMA_LAYERS = 32
ELT = 2  # bf16
# dram__bytes_read.sum + dram__bytes_write.sum of one paged_attention_decode_fused call on this
# workload with separate pools and the per-partition grid (partition kernel 578.7 + 2.9 MB, merge
# kernel 4.3 MB with the cold L2 of the capture; mean of two calls), from one ncu capture of those
# metrics on the current kernels (no sleep between barrier polls).  Retake it whenever either
# kernel changes.
FUSED_CALL_DRAM_BYTES = 585.9e6
# dram__bytes_read.sum + dram__bytes_write.sum of one tcgen05 prefill launch on the chunked-prefill
# workload (554.4 + 235.2 MB, mean of two launches), from one ncu capture of those metrics on the
# current kernel (K 2 / V 3 rings, no sleep between barrier polls).  Retake it whenever the kernel
# changes.
PREFILL_DRAM_BYTES = 789.6e6


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def algorithmic_bytes(lens, batch):
    """Bytes the step must move at minimum: K and V of exactly context_len tokens per sequence and
    KV head, the queries and outputs, the table entries and lengths read, and the write (new K/V
    read once, written once, plus slots)."""
    kv = sum(lens) * HKV * D * ELT * 2
    qo = 2 * batch * HQ * D * ELT
    tables = sum(W.ceil_div(n, S) for n in lens) * 4 + batch * 4
    write = batch * HKV * D * ELT * 2 * 2 + batch * 8
    return kv + qo + tables, write


class ClockSampler:
    """nvidia-smi samples during the timed region (clocks and throttle reasons)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        return rank, world, local, dist
    if n_gpus > 1:
        print(json.dumps({"warning": "--gpus > 1 without torchrun; running one replica"}), file=sys.stderr)
    return 0, 1, 0, None


def barrier(dist, cuda: bool = True):
    if dist is not None:
        dist.barrier()
    if cuda:
        torch.cuda.synchronize()


def max_over_ranks(x: float, dist, device: str = "cuda") -> float:
    """The slowest rank's time: every replica's timed region counts in full."""
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_seed(rank: int) -> int:
    """Each replica draws its own device inputs (same shapes, different values)."""
    return W.SEED_BASE + 3 + 1000 * rank


def whole_job_gbs(step_bytes: float, steps: int, world: int, slowest_ms: float) -> float:
    """Weak scaling: every replica moves step_bytes per step; the job's throughput is all replicas'
    bytes over the slowest replica's time."""
    return step_bytes * steps * world / (slowest_ms * 1e-3) / 1e9


def cpu_baseline(budget_s: float = 10.0):
    """The oracle (fp64 numpy, gather + explicit repeat + two-pass softmax), as it stands, on the
    host cores, over the sequences of the same serving batch (write + decode per sequence, cycling)
    until about ``budget_s`` seconds of oracle time are spent."""
    import oracle
    lens = W.llama_context_lens()
    threads = torch.get_num_threads()
    torch.set_num_threads(1)  # the oracle's torch indexing on one core, like its numpy arithmetic
    done_bytes, spent, seqs, tokens = 0, 0.0, 0, 0
    g_bytes, g_spent = 0, 0.0
    while spent < budget_s and seqs < 512:
        n = lens[seqs % len(lens)]
        case = W.decode_case("cpu_sample", W.SEED_BASE + 3 + 17 * seqs, [n - 1], n_q_heads=HQ, n_kv_heads=HKV,
                             head_dim=D, block_size=S, dtype=torch.bfloat16,
                             num_blocks=W.ceil_div(n, S) + 1, max_blocks_per_seq=W.LLAMA_MAX_CTX // S)
        t0 = time.perf_counter()
        kp, vp = oracle.paged_kv_write(case.k_pool, case.v_pool, case.k_new, case.v_new, case.slot_mapping)
        oracle.paged_decode(case.q, kp, vp, case.block_table, case.context_lens, case.scale)
        spent += time.perf_counter() - t0
        # the gather alone: the contiguous copy of K and V through the block table that a fused
        # paged read avoids
        t1 = time.perf_counter()
        oracle.gather_history(kp, case.block_table[0], n, S)
        oracle.gather_history(vp, case.block_table[0], n, S)
        g_spent += time.perf_counter() - t1
        g_bytes += n * HKV * D * ELT * 2
        kvb, wb = algorithmic_bytes([n], 1)
        done_bytes += kvb + wb
        tokens += n
        seqs += 1
    torch.set_num_threads(threads)
    return {"value": done_bytes / spent / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{seqs} sequences of the 64-sequence serving batch, cycled (write + decode, {tokens} "
                      f"context tokens), {spent:.1f} s of single-threaded numpy / torch fp64",
            "gather_only": {"value": g_bytes / g_spent / 1e9, "unit": UNIT,
                            "what": "the oracle's contiguous gather of each sequence's K and V through its block "
                                    "table (upcast to fp64), alone: the copy the fused paged read avoids"}}


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on the host cores.  Each step is a bounded
    sample of the serving step: the write of one sequence's new token and the decode attention of
    one (sequence, KV head) row of it (G = 4 query heads over its whole context), rotating over
    sequences and heads."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    torch.set_num_threads(1)  # one host core, as the line states
    lens = W.llama_context_lens()
    cases = []
    for i in range(8):
        n = lens[i]
        cases.append((n, W.decode_case("ref_sample", W.SEED_BASE + 3 + i, [n - 1], n_q_heads=HQ, n_kv_heads=HKV,
                                       head_dim=D, block_size=S, dtype=torch.bfloat16,
                                       num_blocks=W.ceil_div(n, S) + 1, max_blocks_per_seq=W.LLAMA_MAX_CTX // S)))

    def step(i):
        n, c = cases[i % len(cases)]
        kvh = (i // len(cases)) % HKV
        kp, vp = oracle.paged_kv_write(c.k_pool, c.v_pool, c.k_new, c.v_new, c.slot_mapping)
        oracle.paged_decode_rows(c.q, kp, vp, c.block_table, c.context_lens, c.scale, [(0, kvh)])
        kvb, wb = algorithmic_bytes([n], 1)
        return (kvb + wb) / HKV

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    total = 0.0
    for i in range(args.steps):
        total += step(i)
    dt = time.perf_counter() - t0
    value = total / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) K/V/Q, bf16-cast, upcast to fp64)",
            "config": {"workload": "llama3_8b_serving_decode sample: per step the write + decode of one "
                                   "(sequence, KV head) row of the batch-64 U[512,4096] serving step",
                       "heads": "32q/8kv", "head_dim": D, "block_size": S},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": "one (sequence, KV head) row per step, rotating over 8 sequences x 8 heads"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def prefill_flops(case) -> float:
    """Unmasked (query, key) pairs x 4 x head_dim x query heads (QK^T and PV, 2 flops per MAC)."""
    qsl = case.query_start_loc.tolist()
    lens = case.context_lens.tolist()
    pairs = 0
    for b in range(len(lens)):
        m = qsl[b + 1] - qsl[b]
        n = lens[b]
        pairs += m * (n - m) + m * (m + 1) // 2
    return 4.0 * case.head_dim * case.n_q_heads * pairs


def run_prefill(args):
    """Chunked-prefill workload: 128 sequences over a 1024-token shared prefix, suffixes U[0,512],
    chunks of 256 queries; one step = paged_kv_write of the 32,768 chunk tokens + causal prefill."""
    import pagedattention_kv_cache_paged_gb300 as pa
    lib = pa.load_library()
    pa.set_option(pa.PA_OPT_PREFILL_KERNEL, args.prefill_kernel)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    case = W.prefill_cow()
    kp, vp = case.k_pool.to(dev), case.v_pool.to(dev)
    q, kn, vn = case.q.to(dev), case.k_new.to(dev), case.v_new.to(dev)
    slot, table = case.slot_mapping.to(dev), case.block_table.to(dev)
    ctx, qsl = case.context_lens.to(dev), case.query_start_loc.to(dev)
    out = torch.empty_like(q)
    NB, S, Hkv, Dh = kp.shape
    T = int(slot.numel())
    flops = prefill_flops(case)

    def step():
        st = lib.paged_kv_write(kn.data_ptr(), vn.data_ptr(), slot.data_ptr(), T, kp.data_ptr(), vp.data_ptr(),
                                NB, S, Hkv, Dh, pa.PA_BF16, sp)
        if st:
            raise RuntimeError(f"paged_kv_write status {st}")
        ev[0].record(stream)
        st = lib.paged_attention_prefill(out.data_ptr(), q.data_ptr(), qsl.data_ptr(), q.shape[0], kp.data_ptr(),
                                         vp.data_ptr(), table.data_ptr(), table.stride(0), ctx.data_ptr(),
                                         ctx.numel(), NB, S, case.scale, case.n_q_heads, Hkv, Dh, pa.PA_BF16, sp)
        if st:
            raise RuntimeError(f"paged_attention_prefill status {st}")
        ev[1].record(stream)

    ev = [torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
    for _ in range(args.warmup):
        step()
    K = args.steps
    pf_ms = []
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(0)
    torch.cuda.synchronize()
    launches0 = pa.launch_count()
    clocks.start()
    ev0.record(stream)
    for _ in range(K):
        step()
        torch.cuda.synchronize()
        pf_ms.append(ev[0].elapsed_time(ev[1]))
    ev1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    launches = pa.launch_count() - launches0
    total_ms = ev0.elapsed_time(ev1)
    pf = statistics.median(pf_ms)
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {"bf16_tflops": 1900.0}
    peak = float(peaks["bf16_tflops"])
    if pa.device_error_flags() != 0:
        raise RuntimeError("device error word set during the benchmark")
    line = {
        "metric": "paged chunked prefill: TFLOP/s over unmasked pairs", "value": flops / (pf * 1e-3) / 1e12,
        "unit": "TFLOP/s", "n_gpus": 1, "steps": K, "warmup": args.warmup, "ms_per_step": total_ms / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) Q/K/V, bf16)",
        "config": {"workload": "chunked prefill: 128 seqs, 1024-token shared prefix (32 blocks of 32, refcount "
                               "128), suffix U[0,512], causal chunk of 256, 32q/8kv heads, head_dim 128",
                   "prefill_kernel": ["auto (tcgen05)", "cuda-core", "tcgen05", "mma.sync"][args.prefill_kernel],
                   "gflop_per_step": flops / 1e9, "steps_synchronised": True,
                   "l2": "inputs larger than L2: per step 268 MB of queries, 134 MB of chunk K/V written, "
                         "a 537 MB pool read"},
        "kernel_us": {"prefill_median": pf * 1e3, "step_incl_write": total_ms / K * 1e3},
        "roofline": {"bound": "tensor", "kernel": "paged_attention_prefill", "achieved": flops / (pf * 1e-3) / 1e12,
                     "peak": peak, "peak_kind": "measured bf16 dense (burst)", "unit": "TFLOP/s",
                     "frac": flops / (pf * 1e-3) / 1e12 / peak,
                     "traffic": PREFILL_DRAM_BYTES if args.prefill_kernel in (0, 2) else None},
        "gpu_launches": launches, "clocks": clk,
    }
    print(json.dumps(line))
    return 0


def _timed_fused_decode(pa, lib, *, lens, Hq, Hkv, Dh, S, dtype, code, pools_count, num_blocks, max_blocks, reps,
                        warmup, seed, flush_bytes, graph=False):
    """Median device time of one paged_attention_decode_fused call (CUDA events around the call on
    its stream), over ``reps`` calls that rotate through ``pools_count`` independent pools, with an
    L2 flush (a write of ``flush_bytes``) between calls when that is non-zero.  With ``graph``, also
    the median time per call of a CUDA graph holding one call per pool (a captured layer loop),
    replayed ``reps`` times with the flush before each replay: (single-call ms, per-call ms in the
    graph)."""
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    inp = W.device_decode_inputs(lens, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=Dh, block_size=S, dtype=dtype,
                                 num_blocks=num_blocks, max_blocks_per_seq=max_blocks, device=dev, seed=seed,
                                 layers=pools_count)
    table, ctx, slot = inp["block_table"].to(dev), inp["context_lens"].to(dev), inp["slot_mapping"].to(dev)
    q, kn, vn = inp["q"].to(dev), inp["k_new"].to(dev), inp["v_new"].to(dev)
    out = torch.empty_like(q)
    B = len(lens)
    ws_bytes = pa.decode_workspace_size(B, table.stride(0), S, Hq, Hkv, Dh)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    flush = torch.empty(max(flush_bytes // 4, 1), dtype=torch.float32, device=dev) if flush_bytes else None
    scale = 1.0 / math.sqrt(Dh)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def call(i):
        kp, vp = inp["pools"][i % pools_count]
        st = lib.paged_attention_decode_fused(out.data_ptr(), q.data_ptr(), kn.data_ptr(), vn.data_ptr(),
                                              slot.data_ptr(), kp.data_ptr(), vp.data_ptr(), table.data_ptr(),
                                              table.stride(0), ctx.data_ptr(), B, num_blocks, S, scale, Hq, Hkv, Dh,
                                              code, ws.data_ptr(), ws_bytes, sp)
        if st:
            raise RuntimeError(f"paged_attention_decode_fused status {st}")

    times = []
    for i in range(warmup + reps):
        if flush is not None:
            flush.fill_(float(i))
        e0.record(stream)
        call(i)
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= warmup:
            times.append(e0.elapsed_time(e1))
    if not graph:
        del inp
        return statistics.median(times)
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for i in range(pools_count):
            kp, vp = inp["pools"][i]
            st = lib.paged_attention_decode_fused(out.data_ptr(), q.data_ptr(), kn.data_ptr(), vn.data_ptr(),
                                                  slot.data_ptr(), kp.data_ptr(), vp.data_ptr(), table.data_ptr(),
                                                  table.stride(0), ctx.data_ptr(), B, num_blocks, S, scale, Hq, Hkv,
                                                  Dh, code, ws.data_ptr(), ws_bytes, side.cuda_stream)
            if st:
                raise RuntimeError(f"paged_attention_decode_fused status {st} under capture")
    torch.cuda.synchronize()
    gtimes = []
    for i in range(warmup + reps):
        if flush is not None:
            flush.fill_(float(i))
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= warmup:
            gtimes.append(e0.elapsed_time(e1) / pools_count)
    del g, inp
    return statistics.median(times), statistics.median(gtimes)


def run_long(args):
    """Long-context split-K decode: batch 4 at 32K/64K/96K/128K tokens, 32 query / 8 KV heads,
    head_dim 128, block_size 16, bf16; one step = one fused write + decode call (the split-K
    partition kernel and the log-sum-exp merge).  Inputs are larger than L2 (1.34 GB of K/V per
    call, two rotating pools)."""
    import pagedattention_kv_cache_paged_gb300 as pa
    lib = pa.load_library()
    pa.set_option(pa.PA_OPT_PARTITION_TOKENS, args.partition_tokens)
    pa.set_option(pa.PA_OPT_DECODE_GRID, args.decode_grid)
    lens = list(W.LONG_LENS)
    need = sum(W.ceil_div(n, S) for n in lens)
    nb = W.ceil_div(5 * need, 4)
    clocks = ClockSampler(0)
    launches0 = pa.launch_count()
    clocks.start()
    ms = _timed_fused_decode(pa, lib, lens=lens, Hq=HQ, Hkv=HKV, Dh=D, S=S, dtype=torch.bfloat16, code=pa.PA_BF16,
                             pools_count=2, num_blocks=nb, max_blocks=W.ceil_div(max(lens), S), reps=args.steps,
                             warmup=args.warmup, seed=SEED_LONG, flush_bytes=0)
    clk = clocks.stop()
    launches = pa.launch_count() - launches0
    kvb, wb = algorithmic_bytes(lens, len(lens))
    gbs = (kvb + wb) / (ms * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    if pa.device_error_flags() != 0:
        raise RuntimeError("device error word set during the benchmark")
    line = {
        "metric": METRIC, "value": gbs, "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) Q/K/V, bf16)",
        "config": {"workload": "long_context_split_k_decode: batch 4 at 32768/65536/98304/131072 tokens, 32q/8kv "
                               "heads, head_dim 128, block_size 16, write + decode in one fused call",
                   "context_tokens": sum(lens), "l2": "inputs larger than L2: 1.34 GB of K/V per call, 2 pools",
                   "partition_tokens": args.partition_tokens or "auto (1024 at this shape)",
                   "decode_grid": ["one CTA per partition", "equal work per warp"][args.decode_grid],
                   "timing": "median of per-call CUDA events"},
        "pct_hbm_measured": gbs / peak,
        "decode_tok_s_attention_only": len(lens) / (LLAMA_LAYERS * ms * 1e-3),
        "roofline": {"bound": "hbm", "kernel": "paged_attention_decode_fused (partition + merge kernels)",
                     "achieved": gbs, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": gbs / peak,
                     "traffic": None},
        "gpu_launches": launches, "clocks": clk,
    }
    print(json.dumps(line))
    return 0


def run_gpt2(args):
    """GPT-2-small-shaped decode sweep: 12 query = 12 KV heads, head_dim 64, block_size 16, fp16;
    batch {1, 2, 4, 8} x context {128 .. 2048}; per cell the median device time of one layer's fused
    write + decode call over 12 layer pools, with an L2 flush between calls (most cells fit in L2
    and are launch-bound: their time is reported in us)."""
    import pagedattention_kv_cache_paged_gb300 as pa
    lib = pa.load_library()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    cells = []
    peak, peak_kind = measured_peaks()
    clocks = ClockSampler(0)
    launches0 = pa.launch_count()
    clocks.start()
    for bi, batch in enumerate(W.GPT2_BATCHES):
        for ci, context in enumerate(W.GPT2_CONTEXTS):
            lens = [context] * batch
            need = batch * W.ceil_div(context, 16)
            ms, gms = _timed_fused_decode(pa, lib, lens=lens, Hq=12, Hkv=12, Dh=64, S=16, dtype=torch.float16,
                                          code=pa.PA_FP16, pools_count=W.GPT2_LAYERS,
                                          num_blocks=W.ceil_div(5 * need, 4), max_blocks=W.ceil_div(context, 16),
                                          reps=args.steps, warmup=args.warmup, seed=W.SEED_BASE + 2 + 31 * bi + ci,
                                          flush_bytes=2 * l2, graph=True)
            kv = batch * context * 12 * 64 * 2 * 2
            qo = 2 * batch * 12 * 64 * 2
            wb = batch * 12 * 64 * 2 * 2 * 2
            gbs = (kv + qo + wb) / (ms * 1e-3) / 1e9
            cells.append({"batch": batch, "context": context, "us_per_layer_call": ms * 1e3, "GB/s": gbs,
                          "tok_s_attention_only_12_layers": batch / (W.GPT2_LAYERS * ms * 1e-3),
                          "us_per_layer_in_12_layer_graph": gms * 1e3,
                          "GB/s_in_graph": (kv + qo + wb) / (gms * 1e-3) / 1e9})
    clk = clocks.stop()
    launches = pa.launch_count() - launches0
    if pa.device_error_flags() != 0:
        raise RuntimeError("device error word set during the benchmark")
    big = cells[-1]
    line = {
        "metric": METRIC, "value": big["GB/s"], "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": big["us_per_layer_call"] / 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp16", "data": "synthetic (seeded N(0,1) Q/K/V, fp16)",
        "config": {"workload": "gpt2_small_decode_sweep: 12q = 12kv heads, head_dim 64, block_size 16, fp16, "
                               "batch {1,2,4,8} x context {128..2048}, 12 layer pools; value = batch 8 x 2048",
                   "l2": "L2 flushed (write of 2x L2) before every timed call or graph replay",
                   "timing": "median of per-call CUDA events; also a CUDA graph of the 12 layers' calls, replayed, per call"},
        "cells": cells,
        "roofline": {"bound": "hbm", "kernel": "paged_attention_decode_fused at batch 8 x 2048 (50 MB per call)",
                     "achieved": big["GB/s"], "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": big["GB/s"] / peak, "traffic": None},
        "gpu_launches": launches, "clocks": clk,
    }
    print(json.dumps(line))
    return 0


def run_swap(args):
    """Block swap between the device pool and a pinned host pool (the offload tier): 8192 blocks of the
    serving shape (32 KB of K and 32 KB of V each, 512 MB per direction) swapped out, then swapped
    back in to other physical blocks, one swap_blocks call per direction."""
    import pagedattention_kv_cache_paged_gb300 as pa
    lib = pa.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    NB, NH = W.LLAMA_POOL, 8192
    gen = torch.Generator(device=dev)
    gen.manual_seed(W.SEED_BASE + 6)
    kp = torch.randn((NB, S, HKV, D), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
    vp = torch.randn((NB, S, HKV, D), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
    hk = torch.empty((NH, S, HKV, D), dtype=torch.bfloat16).pin_memory()
    hv = torch.empty((NH, S, HKV, D), dtype=torch.bfloat16).pin_memory()
    hgen = torch.Generator().manual_seed(W.SEED_BASE + 6)
    perm = torch.randperm(NB, generator=hgen)
    out_pairs = torch.stack([perm[:NH], torch.arange(NH)], dim=1).to(torch.int64).to(dev)
    in_pairs = torch.stack([torch.arange(NH), perm[NH:2 * NH]], dim=1).to(torch.int64).to(dev)
    block_bytes = S * HKV * D * ELT
    moved = NH * block_bytes * 2  # K and V

    def swap(dst, src, pairs, ndst, nsrc):
        st = lib.swap_blocks(dst[0].data_ptr(), dst[1].data_ptr(), ndst, src[0].data_ptr(), src[1].data_ptr(),
                             nsrc, pairs.data_ptr(), NH, block_bytes, sp)
        if st:
            raise RuntimeError(f"swap_blocks status {st}")

    for _ in range(args.warmup):
        swap((hk, hv), (kp, vp), out_pairs, NH, NB)
        swap((kp, vp), (hk, hv), in_pairs, NB, NH)
    K = args.steps
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    t_out, t_in = 0.0, 0.0
    clocks = ClockSampler(0)
    clocks.start()
    launches0 = pa.launch_count()
    for _ in range(K):
        ev[0].record(stream)
        swap((hk, hv), (kp, vp), out_pairs, NH, NB)
        ev[1].record(stream)
        swap((kp, vp), (hk, hv), in_pairs, NB, NH)
        ev[2].record(stream)
        torch.cuda.synchronize()
        t_out += ev[0].elapsed_time(ev[1])
        t_in += ev[1].elapsed_time(ev[2])
    clk = clocks.stop()
    launches = pa.launch_count() - launches0
    if pa.device_error_flags() != 0:
        raise RuntimeError("device error word set during the benchmark")
    line = {"metric": "paged block swap: GB/s between the device pool and a pinned host pool",
            "value": 2 * moved * K / ((t_out + t_in) * 1e-3) / 1e9, "unit": "GB/s", "n_gpus": 1, "steps": K,
            "warmup": args.warmup, "ms_per_step": (t_out + t_in) / K, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "swap_blocks: 8192 blocks x (32 KB K + 32 KB V) device -> pinned host, then "
                                   "host -> device into other blocks (Llama-3-8B pool shape)",
                       "bytes_per_direction": moved,
                       "l2": "inputs larger than L2: 537 MB moved each way per step"},
            "swap_out_gbs": moved * K / (t_out * 1e-3) / 1e9, "swap_in_gbs": moved * K / (t_in * 1e-3) / 1e9,
            "gpu_launches": launches, "clocks": clk}
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=4, help="independent layer pools rotated over the steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=1000)
    ap.add_argument("--partition-tokens", type=int, default=0, help="split-K partition length (0 = library default)")
    ap.add_argument("--decode-kernel", type=int, default=0, help="0 auto, 1 CUDA-core, 2 tensor-core")
    ap.add_argument("--decode-grid", type=int, default=0,
                    help="split-K grid of the tensor-core decode: 0 one CTA per partition, 1 equal work per warp")
    ap.add_argument("--workload", choices=["decode", "prefill", "swap", "long", "gpt2"], default="decode")
    ap.add_argument("--unfused", action="store_true",
                    help="time paged_kv_write + paged_attention_decode as two calls instead of the fused call")
    ap.add_argument("--prefill-kernel", type=int, default=0, help="0 auto, 1 CUDA-core, 2 tcgen05, 3 mma.sync")
    ap.add_argument("--kv-layout", choices=["separate", "unified"], default="separate",
                    help="separate K and V pools, or one pool of unified K/V blocks")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "prefill":
        return run_prefill(args)
    if args.workload == "swap":
        return run_swap(args)
    if args.workload == "long":
        return run_long(args)
    if args.workload == "gpt2":
        return run_gpt2(args)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    rank, world, local, dist = dist_setup(args.gpus)
    import pagedattention_kv_cache_paged_gb300 as pa
    lib = pa.load_library()
    pa.set_option(pa.PA_OPT_PARTITION_TOKENS, args.partition_tokens)
    pa.set_option(pa.PA_OPT_DECODE_KERNEL, args.decode_kernel)
    pa.set_option(pa.PA_OPT_DECODE_GRID, args.decode_grid)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream

    lens = W.llama_context_lens()
    B = len(lens)
    inp = W.device_decode_inputs(lens, n_q_heads=HQ, n_kv_heads=HKV, head_dim=D, block_size=S,
                                 dtype=torch.bfloat16, num_blocks=W.LLAMA_POOL,
                                 max_blocks_per_seq=W.LLAMA_MAX_CTX // S, device=dev,
                                 seed=replica_seed(rank), layers=args.layers)
    table = inp["block_table"].to(dev)
    ctx = inp["context_lens"].to(dev)
    slot = inp["slot_mapping"].to(dev)
    q = inp["q"].to(dev)
    kn, vn = inp["k_new"].to(dev), inp["v_new"].to(dev)
    out = torch.empty_like(q)
    bt_stride = table.stride(0)
    ws_bytes = pa.decode_workspace_size(B, bt_stride, S, HQ, HKV, D)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(D)
    pools = inp["pools"]
    if args.kv_layout == "unified":
        pa.set_option(pa.PA_OPT_KV_LAYOUT, pa.KV_LAYOUT_UNIFIED)
        unified = []
        for i in range(len(pools)):
            kp, vp = pools[i]
            pools[i] = None
            u = torch.stack([kp, vp], dim=1)
            del kp, vp
            unified.append(u)
            pools[i] = pa.unified_views(u)
    ptr = {k: v.data_ptr() for k, v in dict(table=table, ctx=ctx, slot=slot, q=q, kn=kn, vn=vn, out=out,
                                            ws=ws).items()}

    def write(layer):
        kp, vp = pools[layer]
        st = lib.paged_kv_write(ptr["kn"], ptr["vn"], ptr["slot"], B, kp.data_ptr(), vp.data_ptr(),
                                W.LLAMA_POOL, S, HKV, D, pa.PA_BF16, sp)
        if st:
            raise RuntimeError(f"paged_kv_write status {st}")

    def decode(layer):
        kp, vp = pools[layer]
        st = lib.paged_attention_decode(ptr["out"], ptr["q"], kp.data_ptr(), vp.data_ptr(), ptr["table"],
                                        bt_stride, ptr["ctx"], B, W.LLAMA_POOL, S, scale, HQ, HKV, D,
                                        pa.PA_BF16, ptr["ws"], ws_bytes, sp)
        if st:
            raise RuntimeError(f"paged_attention_decode status {st}")

    def fused(layer):
        kp, vp = pools[layer]
        st = lib.paged_attention_decode_fused(ptr["out"], ptr["q"], ptr["kn"], ptr["vn"], ptr["slot"], kp.data_ptr(),
                                              vp.data_ptr(), ptr["table"], bt_stride, ptr["ctx"], B, W.LLAMA_POOL, S,
                                              scale, HQ, HKV, D, pa.PA_BF16, ptr["ws"], ws_bytes, sp)
        if st:
            raise RuntimeError(f"paged_attention_decode_fused status {st}")

    use_fused = not args.unfused

    def step_pre(layer):
        if not use_fused:
            write(layer)

    def step_main(layer):
        if use_fused:
            fused(layer)
        else:
            decode(layer)

    for i in range(args.warmup):
        step_pre(i % args.layers)
        step_main(i % args.layers)
    K = args.steps
    TIME_EVERY = 8  # the decode call of every 8th step is bracketed by events (fewer records, less overhead)
    ev_dec = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range((K + TIME_EVERY - 1) // TIME_EVERY)]
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier(dist)
    launches0 = pa.launch_count()
    clocks.start()
    ev0.record(stream)
    for i in range(K):
        layer = i % args.layers
        step_pre(layer)
        if i % TIME_EVERY == 0:
            ev_dec[i // TIME_EVERY][0].record(stream)
            step_main(layer)
            ev_dec[i // TIME_EVERY][1].record(stream)
        else:
            step_main(layer)
    ev1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(dist)
    launches = pa.launch_count() - launches0
    total_ms = max_over_ranks(ev0.elapsed_time(ev1), dist)
    dec_ms = statistics.mean(a.elapsed_time(b) for a, b in ev_dec)
    kvb, wb = algorithmic_bytes(lens, B)
    step_bytes = kvb + wb
    ms_per_step = total_ms / K
    value = whole_job_gbs(step_bytes, K, world, total_ms)
    peak, peak_kind = measured_peaks()
    achieved = (step_bytes if use_fused else kvb) / (dec_ms * 1e-3) / 1e9
    if pa.device_error_flags() != 0:
        raise RuntimeError("device error word set during the benchmark")

    # end to end through the C ABI with pinned host buffers: every step copies its inputs (queries,
    # new K/V, slots, tables, lengths) host -> device and its output device -> host.  Two buffer sets
    # and three streams let step i + 1's upload and step i - 1's download run under step i's kernels.
    e2e = None
    E = args.e2e_steps
    if E > 0:
        names = ("q", "kn", "vn", "slot", "table", "ctx")
        src = dict(q=q, kn=kn, vn=vn, slot=slot, table=table, ctx=ctx)
        host = {k: src[k].cpu().pin_memory() for k in names}
        host_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        sets = [{k: torch.empty_like(src[k]) for k in names} for _ in range(2)]
        for st_ in sets:
            st_["out"] = torch.empty_like(out)
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = host_out[0].numel() * host_out[0].element_size()
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        in_ready = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        freed = [torch.cuda.Event() for _ in range(2)]

        def e2e_step(i):
            j = i & 1
            bufs = sets[j]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(freed[j])
                for k in names:
                    bufs[k].copy_(host[k], non_blocking=True)
                in_ready[j].record(s_in)
            stream.wait_event(in_ready[j])
            kp, vp = pools[i % args.layers]
            st = lib.paged_attention_decode_fused(bufs["out"].data_ptr(), bufs["q"].data_ptr(), bufs["kn"].data_ptr(),
                                                  bufs["vn"].data_ptr(), bufs["slot"].data_ptr(), kp.data_ptr(),
                                                  vp.data_ptr(), bufs["table"].data_ptr(), bt_stride,
                                                  bufs["ctx"].data_ptr(), B, W.LLAMA_POOL, S, scale, HQ, HKV, D,
                                                  pa.PA_BF16, ptr["ws"], ws_bytes, sp)
            if st:
                raise RuntimeError(f"paged_attention_decode_fused status {st}")
            done[j].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done[j])
                host_out[j].copy_(bufs["out"], non_blocking=True)
                freed[j].record(s_out)

        for i in range(4):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier(dist)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for i in range(E):
            e2e_step(i)
        e1.record(s_out)
        torch.cuda.synchronize()
        barrier(dist)
        e_ms = max_over_ranks(e0.elapsed_time(e1), dist)
        e2e = {"value": whole_job_gbs(step_bytes, E, world, e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms / E,
               "api": "paged_attention_decode_fused through the C ABI, pinned host buffers, copies overlapped "
                      "with the previous/next step on two copy streams"}

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) Q/K/V, bf16)",
        "config": {"workload": "llama3_8b_serving_decode: write of the 64 new tokens through slot_mapping + paged "
                               "decode attention (" + ("one fused call" if use_fused else "two calls") + "), "
                               "32q/8kv heads, head_dim 128, block_size 16, batch 64, context U[512,4096], "
                               "40,000-block shuffled pool",
                   "context_tokens": sum(lens), "batch": B,
                   "l2": f"inputs larger than L2: {args.layers} rotating layer pools, "
                         f"{kvb / 1e6:.0f} MB of K/V read per step",
                   "parallelism": f"replicas x{world}",
                   "partition_tokens": args.partition_tokens or "auto (1024 at this shape)",
                   "decode_kernel": ["auto", "cuda-core", "tensor-core"][args.decode_kernel],
                   "decode_grid": ["one CTA per partition", "equal work per warp"][args.decode_grid],
                   "kv_layout": args.kv_layout},
        "pct_hbm_measured": value / peak,
        "pct_hbm_spec_8000": value / 8000.0,
        "decode_tok_s_attention_only": B * world / (LLAMA_LAYERS * ms_per_step * 1e-3),
        "kernel_us": {"decode_call": dec_ms * 1e3, "step": ms_per_step * 1e3},
        "roofline": {"bound": "hbm",
                     "kernel": ("paged_attention_decode_fused (write + partition kernel, then merge kernel)" if use_fused
                                else "paged_attention_decode (partition + merge kernels)"),
                     "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": achieved / peak,
                     # DRAM bytes of one fused call (both kernels) from the ncu capture; None for the
                     # two-call variant and for the unified layout (not captured)
                     "traffic": (FUSED_CALL_DRAM_BYTES if use_fused and args.kv_layout == "separate"
                                 and args.decode_grid == 0 else None)},
        "gpu_launches": launches,
        "clocks": clk,
        "e2e": e2e,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
