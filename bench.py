"""Benchmark of the paged decode step (KV write + decode attention) at Llama-3-8B GQA shapes.

One step = one layer's pass of the hot path over the serving batch: the write of the 64 new tokens
through ``slot_mapping`` and the decode attention over every sequence's paged context (split-K
partitions and the log-sum-exp merge included), in one fused call — 32 query / 8 KV heads,
head_dim 128, block_size 16, bf16, batch 64, context lengths uniform in [512, 4096], block tables
drawn from a shuffled 40,000-block pool.

Timed on the device with CUDA events around K back-to-back steps after warm-up; steps rotate over
several independent layer pools so that no step finds its K/V in L2 (each step reads ~577 MB; the
rotation spans > 2 GB).  Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle
instead.  Other modes (``--workload``): long-context split-K decode, the GPT-2-shaped sweep, chunked
prefill, the copy-on-write prefill step, the K/V write of a prefill chunk and the block swap.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload ...]
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import threading
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
# dram__bytes_read.sum + dram__bytes_write.sum per launch (or per call of several launches) from one
# ncu capture of those metrics on the current kernels (mean of the captured launches, with the
# capture's cold L2).  Retake them whenever a kernel changes; None = not taken for the current
# kernels.  Serving decode: one paged_attention_decode_fused call (partition + merge kernels).
FUSED_CALL_DRAM_BYTES = 585.72e6
# one tcgen05 prefill launch on the chunked-prefill workload
PREFILL_DRAM_BYTES = 791.66e6
# one decode call (partition + merge) of the GPT-2-shaped batch 8 x 2048 cell
GPT2_8X2048_DRAM_BYTES = 50.52e6
# one paged_kv_write launch of the 32,768-token prefill chunk (the written lines still in L2 when
# the launch ends are written back after it, so the write bytes fall short of the 134 MB written)
WRITE_CHUNK_DRAM_BYTES = 219.82e6
# the copy-on-write step's copy_blocks launch (127 forks of one shared block) and its paged_kv_write
COW_COPY_DRAM_BYTES = 0.147e6
COW_WRITE_DRAM_BYTES = 495.71e6


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def algorithmic_bytes(lens, batch):
    """Bytes the step must move at minimum: K and V of exactly context_len tokens per sequence and
    KV head, the queries and outputs, the table entries and lengths read, and the write (new K/V
    read once, written once, plus slots)."""
    kv = sum(lens) * HKV * D * ELT * 2
    qo = 2 * batch * HQ * D * ELT
    tables = sum(W.ceil_div(n, S) for n in lens) * 4 + batch * 4
    write = batch * HKV * D * ELT * 2 * 2 + batch * 8
    return kv + qo + tables, write


# ------------------------------------------------------------------------------------------------
# clocks during the timed region (read-only)
# ------------------------------------------------------------------------------------------------

class ClockSampler:
    """SM clock and clock-event reasons of one GPU, sampled about every millisecond from start() to
    stop() through NVML (loaded with ctypes; queries only, no setting is touched), so that even a
    timed region of a few milliseconds gets samples.  Falls back to ``nvidia-smi -lms 100`` where
    NVML cannot be loaded.  ``mark(name)`` records host times; stop() reports the samples between
    the marks 'begin' and 'end' (the timed region) next to all samples under load."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}
    NVML_CLOCK_SM = 1

    def __init__(self, index: int):
        self.index = index
        self.samples = []  # (host time, sm MHz, reasons bitmask)
        self.marks = {}
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._smi = None
        self._nvml = None
        self._handle = None

    def _load_nvml(self) -> bool:
        for name in ("libnvidia-ml.so.1", "libnvidia-ml.so"):
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                lib = None
        if lib is None or lib.nvmlInit_v2() != 0:
            return False
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
            return False
        mx = ctypes.c_uint(0)
        if lib.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        self._reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        self._nvml, self._handle = lib, h
        return True

    def _loop(self):
        lib, h = self._nvml, self._handle
        mhz, reasons = ctypes.c_uint(0), ctypes.c_ulonglong(0)
        while not self._stop.is_set():
            t = time.perf_counter()
            if lib.nvmlDeviceGetClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mhz)) == 0:
                r = reasons.value if self._reasons_fn(h, ctypes.byref(reasons)) == 0 else 0
                self.samples.append((t, float(mhz.value), int(r)))
            time.sleep(0.001)

    def start(self):
        try:
            ok = self._load_nvml()
        except (OSError, AttributeError):
            ok = False
        if ok:
            self._thread = threading.Thread(target=self._loop, daemon=True)
            self._thread.start()
            return
        fields = ("index,clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.sw_power_cap")
        try:
            self._smi = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={fields}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self._smi = None

    def mark(self, name: str):
        self.marks[name] = time.perf_counter()

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=2)
            try:
                self._nvml.nvmlShutdown()
            except Exception:
                pass
            samples = self.samples
            source = "NVML every ~1 ms"
        elif self._smi is not None:
            self._smi.terminate()
            try:
                out, _ = self._smi.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self._smi.kill()
                out, _ = self._smi.communicate()
            samples = []
            bits = (0x8, 0x40, 0x20, 0x4)
            for line in out.strip().splitlines():
                parts = [p.strip() for p in line.split(",")]
                try:
                    mhz, self.max_mhz = float(parts[1]), float(parts[2])
                except (ValueError, IndexError):
                    continue
                r = 0
                for bit, v in zip(bits, parts[3:7]):
                    r |= bit if v.lower().startswith("active") else 0
                samples.append((None, mhz, r))
            source = "nvidia-smi every 100 ms"
        else:
            return None
        if not samples:
            return None
        t0, t1 = self.marks.get("begin"), self.marks.get("end")
        timed = [s for s in samples if s[0] is not None and t0 is not None and t1 is not None and t0 <= s[0] <= t1]
        # under load: from the first mark to the last (warm-up, timed region and anything after)
        lo = min(self.marks.values()) if self.marks else None
        hi = max(self.marks.values()) if self.marks else None
        load = [s for s in samples if s[0] is None or lo is None or lo <= s[0] <= hi] or samples
        use = timed if len(timed) >= 3 else load
        reasons = sorted({name for s in use for bit, name in self.REASONS.items() if s[2] & bit})
        return {"sm_mhz": statistics.median(s[1] for s in use), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(use), "samples_timed_region": len(timed),
                "window": "timed region" if use is timed else "warm-up to end of the measured legs",
                "sm_mhz_min": min(s[1] for s in use), "source": source}


# ------------------------------------------------------------------------------------------------
# multi-process (replica) bookkeeping
# ------------------------------------------------------------------------------------------------

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


# ------------------------------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and reference arm)
# ------------------------------------------------------------------------------------------------

_ORACLE_CASES: list = []
_N_ORACLE_CASES = 8


def _serving_sample_case(i: int):
    """Sequence i of the serving batch as a one-sequence case (its history, new token and query)."""
    lens = W.llama_context_lens()
    n = lens[i % len(lens)]
    case = W.decode_case("cpu_sample", W.SEED_BASE + 3 + 17 * i, [n - 1], n_q_heads=HQ, n_kv_heads=HKV, head_dim=D,
                         block_size=S, dtype=torch.bfloat16, num_blocks=W.ceil_div(n, S) + 1,
                         max_blocks_per_seq=W.LLAMA_MAX_CTX // S)
    return n, case


def _oracle_worker_init():
    """Worker process: one host thread (numpy, BLAS and torch), the sample cases built once."""
    torch.set_num_threads(1)
    _ORACLE_CASES.clear()
    _ORACLE_CASES.extend(_serving_sample_case(i) for i in range(_N_ORACLE_CASES))


def _oracle_ready(_):
    return os.getpid()


def _oracle_task(job):
    """One unit of oracle work: ('seq', i) = write + decode of sample sequence i (all heads);
    ('row', i) = write + decode of one (sequence, KV head) row; ('gather', i) = the gather alone.
    Returns (algorithmic bytes, oracle seconds)."""
    import oracle
    kind, i = job
    n, c = _ORACLE_CASES[i % len(_ORACLE_CASES)]
    t0 = time.perf_counter()
    if kind == "gather":
        oracle.gather_history(c.k_pool, c.block_table[0], n, S)
        oracle.gather_history(c.v_pool, c.block_table[0], n, S)
        return n * HKV * D * ELT * 2, time.perf_counter() - t0
    kp, vp = oracle.paged_kv_write(c.k_pool, c.v_pool, c.k_new, c.v_new, c.slot_mapping)
    kvb, wb = algorithmic_bytes([n], 1)
    if kind == "row":
        kvh = (i // len(_ORACLE_CASES)) % HKV
        oracle.paged_decode_rows(c.q, kp, vp, c.block_table, c.context_lens, c.scale, [(0, kvh)])
        return (kvb + wb) / HKV, time.perf_counter() - t0
    oracle.paged_decode(c.q, kp, vp, c.block_table, c.context_lens, c.scale)
    return kvb + wb, time.perf_counter() - t0


class OraclePool:
    """``cores`` worker processes (spawned, one host thread each: the sequence-parallel schedule of
    a CPU kernel that gives each thread whole sequences), their sample cases built before timing."""

    def __init__(self, cores: int):
        import multiprocessing as mp
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"  # inherited by the spawned workers
        self.cores = cores
        self.pool = mp.get_context("spawn").Pool(cores, initializer=_oracle_worker_init)
        self.pool.map(_oracle_ready, range(cores), chunksize=1)

    def run(self, jobs):
        """Wall seconds and algorithmic bytes of the jobs spread over the workers."""
        t0 = time.perf_counter()
        res = self.pool.map(_oracle_task, jobs, chunksize=1)
        return time.perf_counter() - t0, sum(r[0] for r in res)

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_baseline(budget_s: float = 10.0):
    """The oracle (fp64 numpy: gather + explicit repeat + two-pass softmax), as it stands, on the host
    cores over sequences of the serving batch (write + decode per sequence): on a single core for
    about ``budget_s`` seconds of oracle work, then the same number of sequences on every host core
    (one single-threaded worker process per core, each taking whole sequences); plus the oracle's
    gather alone on one core."""
    cores = os.cpu_count() or 1
    runs = []
    one = OraclePool(1)
    try:
        one.run([("seq", 0)])  # the worker's first import of the oracle
        t_seq = one.run([("seq", i) for i in range(_N_ORACLE_CASES)])[0] / _N_ORACLE_CASES
        n_jobs = min(max(int(budget_s / max(t_seq, 1e-3)), 8), 4096)
        secs, nbytes = one.run([("seq", i) for i in range(n_jobs)])
        g_secs, g_bytes = one.run([("gather", i) for i in range(_N_ORACLE_CASES)])
    finally:
        one.close()
    runs.append({"cores": 1, "value": nbytes / secs / 1e9, "unit": UNIT, "sequences": n_jobs, "wall_s": secs})
    if cores > 1:
        pool = OraclePool(cores)
        try:
            pool.run([("seq", i) for i in range(cores)])  # every worker imports the oracle once
            n_all = max(n_jobs, 4 * cores)
            secs, nbytes = pool.run([("seq", i) for i in range(n_all)])
        finally:
            pool.close()
        runs.insert(0, {"cores": cores, "value": nbytes / secs / 1e9, "unit": UNIT, "sequences": n_all,
                        "wall_s": secs})
    best = runs[0]
    return {"value": best["value"], "unit": UNIT, "cores": best["cores"], "kind": "oracle",
            "sample": f"{best['sequences']} sequences of the 64-sequence serving batch (write + decode of every "
                      f"head, {_N_ORACLE_CASES} distinct sequences cycled), spread over {best['cores']} "
                      f"single-threaded numpy / torch fp64 worker processes, {best['wall_s']:.1f} s wall",
            "runs": runs,
            "gather_only": {"value": g_bytes / g_secs / 1e9, "unit": UNIT, "cores": 1,
                            "what": "the oracle's contiguous gather of each sequence's K and V through its block "
                                    "table (upcast to fp64), alone: the copy the fused paged read avoids"}}


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on every host core.  Each step is a bounded
    sample of the serving step: the write of a sequence's new token and the decode attention of one
    (sequence, KV head) row of it (G = 4 query heads over its whole context) on each of the host's
    cores at once (one single-threaded worker process per core), rotating over sequences and
    heads.  A single-core figure of the same rows is reported beside it."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    cores = os.cpu_count() or 1
    pool = OraclePool(cores)
    try:
        for w in range(args.warmup):
            pool.run([("row", w * cores + j) for j in range(cores)])
        total_s, total_b = 0.0, 0.0
        for k in range(args.steps):
            secs, nbytes = pool.run([("row", (args.warmup + k) * cores + j) for j in range(cores)])
            total_s += secs
            total_b += nbytes
    finally:
        pool.close()
    one = OraclePool(1)
    try:
        s1, b1 = one.run([("row", j) for j in range(max(args.steps, 8))])
    finally:
        one.close()
    value = total_b / total_s / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_s / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) K/V/Q, bf16-cast, upcast to fp64)",
            "config": {"workload": "llama3_8b_serving_decode sample: per step the write + decode of one "
                                   "(sequence, KV head) row of the batch-64 U[512,4096] serving step on each "
                                   "host core",
                       "heads": "32q/8kv", "head_dim": D, "block_size": S},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{cores} (sequence, KV head) rows per step, one per single-threaded worker "
                                       f"process, rotating over {_N_ORACLE_CASES} sequences x 8 heads"},
            "cpu_baseline_1core": {"value": b1 / s1 / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
                                   "sample": f"{max(args.steps, 8)} rows on one single-threaded worker"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------------------------------------
# helpers for the GPU modes
# ------------------------------------------------------------------------------------------------

def _opts(pa, **kw):
    return ctypes.byref(pa.make_opts(**kw))


class L2Flush:
    """Evicts the L2 between timed launches: writes a buffer of ``nbytes`` (2x L2 by default), then
    reads a second one of the same size, so that the write's dirty lines are written back here,
    outside the timed region, and not while the next timed kernel streams its own data."""

    def __init__(self, dev, nbytes=None):
        if nbytes is None:
            nbytes = 2 * torch.cuda.get_device_properties(dev).L2_cache_size
        n = max(int(nbytes) // 4, 1)
        self.wbuf = torch.empty(n, dtype=torch.float32, device=dev)
        self.rbuf = torch.zeros(n, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def fill_(self, value):
        self.wbuf.fill_(value)
        torch.sum(self.rbuf, dim=0, out=self.sink)


def _flush_buffer(dev):
    return L2Flush(dev)


def _check_device_flags(pa):
    if pa.device_error_flags() != 0:
        raise RuntimeError("device error word set during the benchmark")


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


def _prefill_device_case(case, dev):
    t = {k: getattr(case, k).to(dev) for k in ("k_pool", "v_pool", "q", "k_new", "v_new", "slot_mapping",
                                               "block_table", "context_lens", "query_start_loc", "copy_pairs")}
    t["out"] = torch.empty_like(t["q"])
    return t


def _launch_write(pa, lib, t, sp, stream_opts=None):
    NB, Sb, Hkv, Dh = t["k_pool"].shape
    T = int(t["slot_mapping"].numel())
    st = lib.paged_kv_write(t["k_new"].data_ptr(), t["v_new"].data_ptr(), t["slot_mapping"].data_ptr(), T,
                            t["k_pool"].data_ptr(), t["v_pool"].data_ptr(), NB, Sb, Hkv, Dh, pa.PA_BF16, sp)
    if st:
        raise RuntimeError(f"paged_kv_write status {st}")


def _launch_prefill(pa, lib, t, case, sp, prefill_kernel=0):
    NB, Sb, Hkv, Dh = t["k_pool"].shape
    st = lib.paged_attention_prefill_ex(t["out"].data_ptr(), t["q"].data_ptr(), t["query_start_loc"].data_ptr(),
                                        t["q"].shape[0], t["k_pool"].data_ptr(), t["v_pool"].data_ptr(),
                                        t["block_table"].data_ptr(), t["block_table"].stride(0),
                                        t["context_lens"].data_ptr(), t["context_lens"].numel(), NB, Sb, case.scale,
                                        case.n_q_heads, Hkv, Dh, pa.PA_BF16, _opts(pa, prefill_kernel=prefill_kernel),
                                        sp)
    if st:
        raise RuntimeError(f"paged_attention_prefill status {st}")


def _launch_copy(pa, lib, t, sp):
    NB, Sb, Hkv, Dh = t["k_pool"].shape
    n = int(t["copy_pairs"].shape[0])
    st = lib.copy_blocks(t["k_pool"].data_ptr(), t["v_pool"].data_ptr(), t["copy_pairs"].data_ptr(), n, NB,
                         Sb * Hkv * Dh * ELT, sp)
    if st:
        raise RuntimeError(f"copy_blocks status {st}")


def _roofline_hbm(achieved, peaks, peak_kind, kernel, traffic=None, per_launch_bytes=None):
    peak = float(peaks["hbm_gbs"])
    r = {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": peak,
         "peak_kind": f"{peak_kind} HBM copy", "unit": "GB/s", "frac": achieved / peak, "traffic": traffic}
    if per_launch_bytes is not None:
        r["algorithmic_bytes_per_launch"] = per_launch_bytes
    return r


# ------------------------------------------------------------------------------------------------
# chunked prefill, copy-on-write step, prefill-chunk write
# ------------------------------------------------------------------------------------------------

def run_prefill(args):
    """Chunked-prefill workload: 128 sequences over a 1024-token shared prefix, suffixes U[0,512],
    chunks of 256 queries; one step = paged_kv_write of the 32,768 chunk tokens + causal prefill.
    The prefill launch is timed with events on its own (median over steps)."""
    import pagedattention_kv_cache_paged_gb300 as pa
    lib = pa.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    case = W.prefill_cow()
    t = _prefill_device_case(case, dev)
    flops = prefill_flops(case)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def step():
        _launch_write(pa, lib, t, sp)
        ev[0].record(stream)
        _launch_prefill(pa, lib, t, case, sp, args.prefill_kernel)
        ev[1].record(stream)

    clocks = ClockSampler(0)
    clocks.start()
    clocks.mark("warmup")
    for _ in range(args.warmup):
        step()
    K = args.steps
    pf_ms = []
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    launches0 = pa.launch_count()
    clocks.mark("begin")
    ev0.record(stream)
    for _ in range(K):
        step()
        torch.cuda.synchronize()
        pf_ms.append(ev[0].elapsed_time(ev[1]))
    ev1.record(stream)
    torch.cuda.synchronize()
    clocks.mark("end")
    clk = clocks.stop()
    launches = pa.launch_count() - launches0
    total_ms = ev0.elapsed_time(ev1)
    pf = statistics.median(pf_ms)
    peaks, kind = measured_peaks()
    peak = float(peaks["bf16_tflops"])
    _check_device_flags(pa)
    tflops = flops / (pf * 1e-3) / 1e12
    line = {
        "metric": "paged chunked prefill: TFLOP/s over unmasked pairs", "value": tflops,
        "unit": "TFLOP/s", "n_gpus": 1, "steps": K, "warmup": args.warmup, "ms_per_step": total_ms / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) Q/K/V, bf16)",
        "config": {"workload": "chunked prefill: 128 seqs, 1024-token shared prefix (32 blocks of 32, refcount "
                               "128), suffix U[0,512], causal chunk of 256, 32q/8kv heads, head_dim 128",
                   "prefill_kernel": ["auto (tcgen05)", "cuda-core", "tcgen05"][args.prefill_kernel],
                   "gflop_per_step": flops / 1e9, "steps_synchronised": True,
                   "l2": "inputs larger than L2: per step 268 MB of queries, 134 MB of chunk K/V written, "
                         "a 537 MB pool read"},
        "kernel_us": {"prefill_median": pf * 1e3, "prefill_min": min(pf_ms) * 1e3,
                      "step_incl_write": total_ms / K * 1e3},
        "roofline": {"bound": "tensor", "kernel": "paged_attention_prefill (tcgen05)", "achieved": tflops,
                     "peak": peak, "peak_kind": f"{kind} bf16 dense (burst)", "unit": "TFLOP/s",
                     "frac": tflops / peak, "frac_of_sustained": tflops / float(peaks.get("bf16_tflops_sustained",
                                                                                         peak)),
                     "traffic": PREFILL_DRAM_BYTES if args.prefill_kernel in (0, 2) else None},
        "gpu_launches": launches, "clocks": clk,
    }
    print(json.dumps(line))
    return 0


def run_cow(args):
    """The copy-on-write arm of the prefill configuration, one step = what a serving engine issues:
    copy_blocks of the 127 forks of the shared partial block (a 1000-token prefix ends inside block
    31), paged_kv_write of every sequence's suffix and chunk, then the causal prefill.  Each call is
    timed with its own events (they are separate launches on one stream, nothing overlaps), the
    pools restored from a pristine copy between steps (untimed)."""
    import pagedattention_kv_cache_paged_gb300 as pa
    lib = pa.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    case = W.prefill_cow(cow_arm=True)
    t = _prefill_device_case(case, dev)
    k0, v0 = t["k_pool"].clone(), t["v_pool"].clone()
    flops = prefill_flops(case)
    NB, Sb, Hkv, Dh = t["k_pool"].shape
    n_pairs = int(case.copy_pairs.shape[0])
    T = int(case.slot_mapping.numel())
    copy_bytes = n_pairs * 2 * 2 * Sb * Hkv * Dh * ELT + n_pairs * 16  # K and V blocks read + written, pairs
    write_bytes = T * Hkv * Dh * ELT * 2 * 2 + T * 8
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    flush = _flush_buffer(dev)

    def step():
        t["k_pool"].copy_(k0)
        t["v_pool"].copy_(v0)
        flush.fill_(1.0)
        ev[0].record(stream)
        _launch_copy(pa, lib, t, sp)
        ev[1].record(stream)
        _launch_write(pa, lib, t, sp)
        ev[2].record(stream)
        _launch_prefill(pa, lib, t, case, sp)
        ev[3].record(stream)
        torch.cuda.synchronize()
        return [ev[i].elapsed_time(ev[i + 1]) for i in range(3)]

    clocks = ClockSampler(0)
    clocks.start()
    clocks.mark("warmup")
    for _ in range(args.warmup):
        step()
    launches0 = pa.launch_count()
    clocks.mark("begin")
    times = [step() for _ in range(args.steps)]
    clocks.mark("end")
    clk = clocks.stop()
    launches = pa.launch_count() - launches0
    _check_device_flags(pa)
    med = [statistics.median(x[i] for x in times) for i in range(3)]
    step_ms = sum(med)
    peaks, kind = measured_peaks()
    tflops = flops / (med[2] * 1e-3) / 1e12
    line = {
        "metric": "paged chunked prefill with copy-on-write forks: TFLOP/s over unmasked pairs per step",
        "value": flops / (step_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) Q/K/V, bf16)",
        "config": {"workload": f"copy-on-write prefill step: {n_pairs} copy_blocks forks of the shared partial "
                               f"block (1000-token prefix, blocks of 32), paged_kv_write of {T} suffix + chunk "
                               "tokens, causal prefill of 128 chunks of 256 queries, 32q/8kv heads, head_dim 128",
                   "l2": "L2 flushed (write of 2x L2, then a read of 2x L2, so that the flush's dirty lines are written back before the timed region) before each step; pools restored before each step (untimed)",
                   "timing": "median per call over the steps, CUDA events between the calls"},
        "kernel_us": {"copy_blocks": med[0] * 1e3, "paged_kv_write": med[1] * 1e3, "prefill": med[2] * 1e3},
        "copy_blocks": {"pairs": n_pairs, "bytes": copy_bytes, "GB/s": copy_bytes / (med[0] * 1e-3) / 1e9,
                        "frac_hbm": copy_bytes / (med[0] * 1e-3) / 1e9 / float(peaks["hbm_gbs"]),
                        "traffic": COW_COPY_DRAM_BYTES,
                        "note": "every fork copies the same shared block (L2-resident after the first): "
                                "launch-latency bound, DRAM traffic far below the bytes copied"},
        "paged_kv_write": {"tokens": T, "bytes": write_bytes, "GB/s": write_bytes / (med[1] * 1e-3) / 1e9,
                           "frac_hbm": write_bytes / (med[1] * 1e-3) / 1e9 / float(peaks["hbm_gbs"]),
                           "traffic": COW_WRITE_DRAM_BYTES},
        "roofline": {"bound": "tensor", "kernel": "paged_attention_prefill (tcgen05)", "achieved": tflops,
                     "peak": float(peaks["bf16_tflops"]), "peak_kind": f"{kind} bf16 dense (burst)",
                     "unit": "TFLOP/s", "frac": tflops / float(peaks["bf16_tflops"]), "traffic": None},
        "gpu_launches": launches, "clocks": clk,
    }
    print(json.dumps(line))
    return 0


def run_write(args):
    """paged_kv_write of the prefill configuration's chunk: 32,768 tokens x 8 KV heads x 128 bf16 of K
    and of V scattered into a 4096-block pool through slot_mapping (268 MB moved: 134 MB read, 134 MB
    written, plus the slots).  Median of per-launch events with an L2 flush before each launch."""
    import pagedattention_kv_cache_paged_gb300 as pa
    lib = pa.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    case = W.prefill_cow()
    t = _prefill_device_case(case, dev)
    NB, Sb, Hkv, Dh = t["k_pool"].shape
    T = int(case.slot_mapping.numel())
    nbytes = T * Hkv * Dh * ELT * 2 * 2 + T * 8
    flush = _flush_buffer(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(0)
    clocks.start()
    clocks.mark("warmup")
    times = []
    launches0 = None
    for i in range(args.warmup + args.steps):
        if i == args.warmup:
            launches0 = pa.launch_count()
            clocks.mark("begin")
        flush.fill_(float(i))
        e0.record(stream)
        _launch_write(pa, lib, t, sp)
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= args.warmup:
            times.append(e0.elapsed_time(e1))
    clocks.mark("end")
    clk = clocks.stop()
    launches = pa.launch_count() - launches0
    _check_device_flags(pa)
    ms = statistics.median(times)
    gbs = nbytes / (ms * 1e-3) / 1e9
    peaks, kind = measured_peaks()
    line = {"metric": "paged_kv_write: GB/s moved (K/V read + written, slots)", "value": gbs, "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) K/V, bf16)",
            "config": {"workload": f"paged_kv_write of the chunked-prefill chunk: {T} tokens x 8 KV heads x 128, "
                                   "block_size 32, 4096-block pool", "bytes_per_launch": nbytes,
                       "l2": "L2 flushed (write of 2x L2, then a read of 2x L2, so that the flush's dirty lines are written back before the timed region) before each launch",
                       "timing": "median of per-launch CUDA events"},
            "roofline": _roofline_hbm(gbs, peaks, kind, "kv_write_kernel", traffic=WRITE_CHUNK_DRAM_BYTES,
                                      per_launch_bytes=nbytes),
            "gpu_launches": launches, "clocks": clk}
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------------------------------------
# decode modes
# ------------------------------------------------------------------------------------------------

def _timed_fused_decode(pa, lib, *, lens, Hq, Hkv, Dh, S, dtype, code, pools_count, num_blocks, max_blocks, reps,
                        warmup, seed, flush_bytes, graph=False, back_to_back=False, partition_tokens=0):
    """Device time of one paged_attention_decode_fused call.  Per-call: the median of CUDA events around
    single calls that rotate through ``pools_count`` independent pools, with an L2 flush (a write
    of ``flush_bytes``, then a read of as many) before each call when that is non-zero.  ``back_to_back``: also the time per
    call of ``reps`` calls issued back to back (events only around the run, so programmatic
    dependent launch overlaps each call with the previous one).  ``graph``: also the median per call
    of a CUDA graph holding one call per pool (a captured layer loop), replayed ``reps`` times with
    the flush before each replay.  Returns a dict of milliseconds."""
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
    ws_bytes = pa.decode_workspace_size(B, table.stride(0), S, Hq, Hkv, Dh, partition_tokens=partition_tokens)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    flush = L2Flush(dev, flush_bytes) if flush_bytes else None
    opts = pa.make_opts(partition_tokens=partition_tokens)
    optp = ctypes.byref(opts)
    scale = 1.0 / math.sqrt(Dh)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def call(i, s=sp):
        kp, vp = inp["pools"][i % pools_count]
        st = lib.paged_attention_decode_fused_ex(out.data_ptr(), q.data_ptr(), kn.data_ptr(), vn.data_ptr(),
                                                 slot.data_ptr(), kp.data_ptr(), vp.data_ptr(), table.data_ptr(),
                                                 table.stride(0), ctx.data_ptr(), B, num_blocks, S, scale, Hq, Hkv,
                                                 Dh, code, ws.data_ptr(), ws_bytes, optp, s)
        if st:
            raise RuntimeError(f"paged_attention_decode_fused status {st}")

    res = {}
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
    res["single"] = statistics.median(times)
    if back_to_back:
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(reps):
            call(i)
        e1.record(stream)
        torch.cuda.synchronize()
        res["back_to_back"] = e0.elapsed_time(e1) / reps
    if graph:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for i in range(pools_count):
                call(i, side.cuda_stream)
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
        res["graph"] = statistics.median(gtimes)
        del g
    del inp
    return res


def run_long(args):
    """Long-context split-K decode: batch 4 at 32K/64K/96K/128K tokens, 32 query / 8 KV heads,
    head_dim 128, block_size 16, bf16; one step = one fused write + decode call (the split-K
    partition kernel and the log-sum-exp merge).  Inputs are larger than L2 (1.34 GB of K/V per
    call, two rotating pools)."""
    import pagedattention_kv_cache_paged_gb300 as pa
    lib = pa.load_library()
    lens = list(W.LONG_LENS)
    need = sum(W.ceil_div(n, S) for n in lens)
    nb = W.ceil_div(5 * need, 4)
    clocks = ClockSampler(0)
    clocks.start()
    clocks.mark("begin")
    launches0 = pa.launch_count()
    r = _timed_fused_decode(pa, lib, lens=lens, Hq=HQ, Hkv=HKV, Dh=D, S=S, dtype=torch.bfloat16, code=pa.PA_BF16,
                            pools_count=2, num_blocks=nb, max_blocks=W.ceil_div(max(lens), S), reps=args.steps,
                            warmup=args.warmup, seed=SEED_LONG, flush_bytes=0, back_to_back=True,
                            partition_tokens=args.partition_tokens)
    clocks.mark("end")
    clk = clocks.stop()
    launches = pa.launch_count() - launches0
    ms = r["single"]
    kvb, wb = algorithmic_bytes(lens, len(lens))
    gbs = (kvb + wb) / (ms * 1e-3) / 1e9
    peaks, kind = measured_peaks()
    _check_device_flags(pa)
    line = {
        "metric": METRIC, "value": gbs, "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) Q/K/V, bf16)",
        "config": {"workload": "long_context_split_k_decode: batch 4 at 32768/65536/98304/131072 tokens, 32q/8kv "
                               "heads, head_dim 128, block_size 16, write + decode in one fused call",
                   "context_tokens": sum(lens), "l2": "inputs larger than L2: 1.34 GB of K/V per call, 2 pools",
                   "timing": "median of per-call CUDA events; back_to_back = per call over a run of calls"},
        "pct_hbm_measured": gbs / float(peaks["hbm_gbs"]),
        "kernel_us": {"call_median": ms * 1e3, "call_back_to_back": r["back_to_back"] * 1e3},
        "decode_tok_s_attention_only": len(lens) / (LLAMA_LAYERS * ms * 1e-3),
        "roofline": _roofline_hbm(gbs, peaks, kind, "paged_attention_decode_fused (partition + merge kernels)",
                                  per_launch_bytes=kvb + wb),
        "gpu_launches": launches, "clocks": clk,
    }
    print(json.dumps(line))
    return 0


def run_gpt2(args):
    """GPT-2-small-shaped decode sweep: 12 query = 12 KV heads, head_dim 64, block_size 16, fp16;
    batch {1, 2, 4, 8} x context {128 .. 2048}; per cell the median device time of one layer's fused
    write + decode call over 12 layer pools, with an L2 flush between calls (most cells fit in L2
    and are launch-bound: their time is reported in us), the per-call time of back-to-back calls,
    and the per-call time inside a CUDA graph of the 12 layers' calls."""
    import pagedattention_kv_cache_paged_gb300 as pa
    lib = pa.load_library()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    cells = []
    peaks, kind = measured_peaks()
    clocks = ClockSampler(0)
    clocks.start()
    clocks.mark("begin")
    launches0 = pa.launch_count()
    only = set(args.gpt2_cells.split(",")) if args.gpt2_cells else None
    for bi, batch in enumerate(W.GPT2_BATCHES):
        for ci, context in enumerate(W.GPT2_CONTEXTS):
            if only is not None and f"{batch}x{context}" not in only:
                continue
            lens = [context] * batch
            need = batch * W.ceil_div(context, 16)
            r = _timed_fused_decode(pa, lib, lens=lens, Hq=12, Hkv=12, Dh=64, S=16, dtype=torch.float16,
                                    code=pa.PA_FP16, pools_count=W.GPT2_LAYERS,
                                    num_blocks=W.ceil_div(5 * need, 4), max_blocks=W.ceil_div(context, 16),
                                    reps=args.steps, warmup=args.warmup, seed=W.SEED_BASE + 2 + 31 * bi + ci,
                                    flush_bytes=2 * l2, graph=True, back_to_back=True,
                                    partition_tokens=args.partition_tokens)
            kv = batch * context * 12 * 64 * 2 * 2
            qo = 2 * batch * 12 * 64 * 2
            wb = batch * 12 * 64 * 2 * 2 * 2
            nbytes = kv + qo + wb
            ms = r["single"]
            cells.append({"batch": batch, "context": context, "bytes": nbytes, "us_per_layer_call": ms * 1e3,
                          "GB/s": nbytes / (ms * 1e-3) / 1e9,
                          "tok_s_attention_only_12_layers": batch / (W.GPT2_LAYERS * ms * 1e-3),
                          "us_per_call_back_to_back": r["back_to_back"] * 1e3,
                          "us_per_layer_in_12_layer_graph": r["graph"] * 1e3,
                          "GB/s_in_graph": nbytes / (r["graph"] * 1e-3) / 1e9})
    clocks.mark("end")
    clk = clocks.stop()
    launches = pa.launch_count() - launches0
    _check_device_flags(pa)
    big = cells[-1]
    line = {
        "metric": METRIC, "value": big["GB/s"], "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": big["us_per_layer_call"] / 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp16", "data": "synthetic (seeded N(0,1) Q/K/V, fp16)",
        "config": {"workload": "gpt2_small_decode_sweep: 12q = 12kv heads, head_dim 64, block_size 16, fp16, "
                               "batch {1,2,4,8} x context {128..2048}, 12 layer pools; value = batch 8 x 2048",
                   "l2": "L2 flushed (write of 2x L2, then a read of 2x L2, so that the flush's dirty lines are written back before the timed region) before every timed single call or graph replay",
                   "timing": "median of per-call CUDA events; per call over back-to-back calls; per call in a "
                             "CUDA graph of the 12 layers' calls, replayed"},
        "cells": cells,
        "roofline": _roofline_hbm(big["GB/s"], peaks, kind,
                                  f"paged_attention_decode_fused at batch {big['batch']} x {big['context']} "
                                  f"({big['bytes'] / 1e6:.1f} MB per call)",
                                  traffic=(GPT2_8X2048_DRAM_BYTES if (big["batch"], big["context"]) == (8, 2048)
                                           and not args.partition_tokens else None),
                                  per_launch_bytes=big["bytes"]),
        "gpu_launches": launches, "clocks": clk,
    }
    print(json.dumps(line))
    return 0


def run_swap(args):
    """Block swap between the device pool and a pinned host pool (the offload tier): 8192 blocks of the
    serving shape (32 KB of K and 32 KB of V each, 512 MB per direction) swapped out, then swapped
    back in to other physical blocks, one swap_blocks call per direction.  The roofline is the host
    link measured in the same run: a contiguous copy of the same bytes between pinned host memory
    and the device (one cudaMemcpyAsync per direction)."""
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

    # the host link alone: the same bytes as one contiguous pinned <-> device copy per direction
    link_h = torch.empty(moved, dtype=torch.uint8).pin_memory()
    link_d = torch.empty(moved, dtype=torch.uint8, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    clocks = ClockSampler(0)
    clocks.start()
    clocks.mark("warmup")
    for _ in range(args.warmup):
        swap((hk, hv), (kp, vp), out_pairs, NH, NB)
        swap((kp, vp), (hk, hv), in_pairs, NB, NH)
        link_h.copy_(link_d, non_blocking=True)
        link_d.copy_(link_h, non_blocking=True)
    torch.cuda.synchronize()
    K = args.steps
    t_out, t_in, c_out, c_in = [], [], [], []
    launches0 = pa.launch_count()
    clocks.mark("begin")
    for _ in range(K):
        ev[0].record(stream)
        swap((hk, hv), (kp, vp), out_pairs, NH, NB)
        ev[1].record(stream)
        swap((kp, vp), (hk, hv), in_pairs, NB, NH)
        ev[2].record(stream)
        torch.cuda.synchronize()
        t_out.append(ev[0].elapsed_time(ev[1]))
        t_in.append(ev[1].elapsed_time(ev[2]))
    launches = pa.launch_count() - launches0
    for _ in range(K):
        ev[0].record(stream)
        link_h.copy_(link_d, non_blocking=True)
        ev[1].record(stream)
        link_d.copy_(link_h, non_blocking=True)
        ev[2].record(stream)
        torch.cuda.synchronize()
        c_out.append(ev[0].elapsed_time(ev[1]))
        c_in.append(ev[1].elapsed_time(ev[2]))
    clocks.mark("end")
    clk = clocks.stop()
    _check_device_flags(pa)
    gb = lambda ms: moved / (ms * 1e-3) / 1e9  # noqa: E731
    so, si = gb(statistics.median(t_out)), gb(statistics.median(t_in))
    lo, li = gb(statistics.median(c_out)), gb(statistics.median(c_in))
    value = 2 * moved / ((statistics.median(t_out) + statistics.median(t_in)) * 1e-3) / 1e9
    link = 2 * moved / ((statistics.median(c_out) + statistics.median(c_in)) * 1e-3) / 1e9
    line = {"metric": "paged block swap: GB/s between the device pool and a pinned host pool",
            "value": value, "unit": "GB/s", "n_gpus": 1, "steps": K,
            "warmup": args.warmup, "ms_per_step": statistics.median(t_out) + statistics.median(t_in),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "swap_blocks: 8192 blocks x (32 KB K + 32 KB V) device -> pinned host, then "
                                   "host -> device into other blocks (Llama-3-8B pool shape)",
                       "bytes_per_direction": moved,
                       "l2": "inputs larger than L2: 537 MB moved each way per step",
                       "timing": "median of per-call CUDA events"},
            "swap_out_gbs": so, "swap_in_gbs": si,
            "host_link": {"d2h_gbs": lo, "h2d_gbs": li, "what": "one contiguous cudaMemcpyAsync of the same "
                                                                  "bytes per direction, pinned host memory"},
            "roofline": {"bound": "host link", "kernel": "swap_blocks_kernel (both directions)", "achieved": value,
                         "peak": link, "peak_kind": "measured pinned host<->device copy, this run", "unit": "GB/s",
                         "frac": value / link, "frac_out": so / lo, "frac_in": si / li, "traffic": None},
            "gpu_launches": launches, "clocks": clk}
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------------------------------------
# the serving decode step (default)
# ------------------------------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=4, help="independent layer pools rotated over the steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=1000)
    ap.add_argument("--partition-tokens", type=int, default=0, help="split-K partition length (0 = library default)")
    ap.add_argument("--decode-kernel", type=int, default=0, help="0 auto, 1 CUDA-core, 2 tensor-core")
    ap.add_argument("--workload", choices=["decode", "prefill", "cow", "write", "swap", "long", "gpt2"],
                    default="decode")
    ap.add_argument("--unfused", action="store_true",
                    help="time paged_kv_write + paged_attention_decode as two calls instead of the fused call")
    ap.add_argument("--gpt2-cells", default="",
                    help="GPT-2 sweep: only these cells, e.g. 8x2048,1x128 (default: all 20)")
    ap.add_argument("--prefill-kernel", type=int, default=0, help="0 auto, 1 CUDA-core, 2 tcgen05")
    ap.add_argument("--kv-layout", choices=["separate", "unified"], default="separate",
                    help="separate K and V pools, or one pool of unified K/V blocks")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    modes = {"prefill": run_prefill, "cow": run_cow, "write": run_write, "swap": run_swap, "long": run_long,
             "gpt2": run_gpt2}
    if args.workload in modes:
        return modes[args.workload](args)

    rank, world, local, dist = dist_setup(args.gpus)
    # the CPU baseline's worker processes are spawned before the first GPU call
    cpu = cpu_baseline() if rank == 0 and not args.no_cpu_baseline else None
    import pagedattention_kv_cache_paged_gb300 as pa
    lib = pa.load_library()
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
    ws_bytes = pa.decode_workspace_size(B, bt_stride, S, HQ, HKV, D, partition_tokens=args.partition_tokens)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(D)
    pools = inp["pools"]
    stride_bytes = 0
    if args.kv_layout == "unified":
        for i in range(len(pools)):
            kp, vp = pools[i]
            pools[i] = None
            u = torch.stack([kp, vp], dim=1)
            del kp, vp
            pools[i] = pa.unified_views(u)
        stride_bytes = 2 * S * HKV * D * ELT
    opts = pa.make_opts(kv_block_stride_bytes=stride_bytes, decode_kernel=args.decode_kernel,
                        partition_tokens=args.partition_tokens)
    optp = ctypes.byref(opts)
    ptr = {k: v.data_ptr() for k, v in dict(table=table, ctx=ctx, slot=slot, q=q, kn=kn, vn=vn, out=out,
                                            ws=ws).items()}

    def write(layer):
        kp, vp = pools[layer]
        st = lib.paged_kv_write_ex(ptr["kn"], ptr["vn"], ptr["slot"], B, kp.data_ptr(), vp.data_ptr(),
                                   W.LLAMA_POOL, S, HKV, D, pa.PA_BF16, optp, sp)
        if st:
            raise RuntimeError(f"paged_kv_write status {st}")

    def decode(layer):
        kp, vp = pools[layer]
        st = lib.paged_attention_decode_ex(ptr["out"], ptr["q"], kp.data_ptr(), vp.data_ptr(), ptr["table"],
                                           bt_stride, ptr["ctx"], B, W.LLAMA_POOL, S, scale, HQ, HKV, D,
                                           pa.PA_BF16, ptr["ws"], ws_bytes, optp, sp)
        if st:
            raise RuntimeError(f"paged_attention_decode status {st}")

    def fused(layer, bufs=None, s=sp):
        kp, vp = pools[layer]
        b = ptr if bufs is None else bufs
        st = lib.paged_attention_decode_fused_ex(b["out"], b["q"], b["kn"], b["vn"], b["slot"], kp.data_ptr(),
                                                 vp.data_ptr(), b["table"], bt_stride, b["ctx"], B, W.LLAMA_POOL,
                                                 S, scale, HQ, HKV, D, pa.PA_BF16, ptr["ws"], ws_bytes, optp, s)
        if st:
            raise RuntimeError(f"paged_attention_decode_fused status {st}")

    use_fused = not args.unfused

    def step(layer):
        if use_fused:
            fused(layer)
        else:
            write(layer)
            decode(layer)

    clocks = ClockSampler(local)
    clocks.start()
    clocks.mark("warmup")
    for i in range(args.warmup):
        step(i % args.layers)
    K = args.steps
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    launches0 = pa.launch_count()
    clocks.mark("begin")
    ev0.record(stream)
    for i in range(K):
        step(i % args.layers)
    ev1.record(stream)
    torch.cuda.synchronize()
    clocks.mark("end")
    barrier(dist)
    launches = pa.launch_count() - launches0
    total_ms = max_over_ranks(ev0.elapsed_time(ev1), dist)
    kvb, wb = algorithmic_bytes(lens, B)
    step_bytes = kvb + wb
    ms_per_step = total_ms / K
    value = whole_job_gbs(step_bytes, K, world, total_ms)
    peaks, peak_kind = measured_peaks()
    # the decode call: in the fused step it is the whole step (K calls back to back, timed together
    # so that each call's partition kernel overlaps the previous call's merge as in serving); the
    # two-call variant times K decode calls back to back after the timed region
    if use_fused:
        dec_ms = ms_per_step
        call_bytes = step_bytes
    else:
        torch.cuda.synchronize()
        ev0.record(stream)
        for i in range(K):
            decode(i % args.layers)
        ev1.record(stream)
        torch.cuda.synchronize()
        dec_ms = ev0.elapsed_time(ev1) / K
        call_bytes = kvb
    achieved = call_bytes / (dec_ms * 1e-3) / 1e9
    _check_device_flags(pa)

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
        set_ptrs = [{k: v.data_ptr() for k, v in st_.items()} for st_ in sets]
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
            fused(i % args.layers, set_ptrs[j])
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
    clocks.mark("after")
    clk = clocks.stop()

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
                   "kv_layout": args.kv_layout,
                   "timing": "CUDA events around the K back-to-back steps"},
        "pct_hbm_measured": value / float(peaks["hbm_gbs"]),
        "pct_hbm_spec_8000": value / 8000.0,
        "decode_tok_s_attention_only": B * world / (LLAMA_LAYERS * ms_per_step * 1e-3),
        "kernel_us": {"decode_call": dec_ms * 1e3, "step": ms_per_step * 1e3},
        "roofline": _roofline_hbm(
            achieved, peaks, peak_kind,
            ("paged_attention_decode_fused: the write + split-K partition kernel and the merge kernel, timed "
             "together because each call's partition kernel overlaps the previous call's merge"
             if use_fused else "paged_attention_decode (partition + merge kernels)"),
            traffic=(FUSED_CALL_DRAM_BYTES if use_fused and args.kv_layout == "separate" else None),
            per_launch_bytes=call_bytes),
        "gpu_launches": launches,
        "clocks": clk,
        "e2e": e2e,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
