#!/usr/bin/env python3
"""Benchmark of the GB300 paged-KV decode engine.

One step = one decode call (split kernel + split-K reduce) over the whole
batch of the workload, inputs resident in HBM, issued as a CUDA-graph
replay. Two device copies of the inputs (one graph each) are alternated so
that no step finds its KV in the 129 MB L2. The append workloads
(append, append_fp8, append_step) time the KV-cache append that precedes a
decode instead: one step = one pa_kv_append(_fp8) call.

    python bench.py [--gpus N] [--steps K] [--warmup W]
                    [--config long|gqa|fp8|tidar|tiny|... (see WORKLOADS)]
                    [--impl ours|reference]

The default workload is the long-context split-K decode (B4, 64/8 heads,
D128, P64, 131072 keys per sequence: 2.15 GB per call), the largest of the
problem statement's workloads that fits one GPU.

Prints one JSON line on rank 0. `value` is the achieved algorithmic HBM
bandwidth in GB/s (bytes a decode must move, see algorithmic_bytes, over
the device time of a call), summed over ranks; `ms_per_step` is the time
of one call. `--impl reference` times the fp64 CPU oracle on all host cores
(one single-threaded process per core, spawned) on a bounded sample of the
same workload; `cpu_baseline` reports that run and a one-core run.
"""

from __future__ import annotations

import os

for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import ctypes
import dataclasses
import hashlib
import json
import math
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from paged_kv_attention_15_gb300 import inputs as gen  # noqa: E402

METRIC = "paged decode µs/call and achieved HBM GB/s (fraction of 8 TB/s) on 1 GB300"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
DEFAULT_CONFIG = "long"

WORKLOADS = {
    "tiny": "tiny paged decode: B2 T1 Hq4 Hkv1 D64 P16 ctx {37,100} bf16",
    "gqa": "GQA decode: B32 T1 Hq32 Hkv8 D128 P16 ctx U[512,8192] bf16",
    "long": "long-context split-K decode: B4 T1 Hq64 Hkv8 D128 P64 ctx 131072 bf16",
    "fp8": "native fp8 KV decode: B64 T1 Hq32 Hkv2 D256 P16 ctx U[1024,16384] e4m3fn KV + fp32 per-token scale",
    "tidar": "TiDAR draft-block decode: B16 T8 Hq32 Hkv8 D128 P16 ctx U[2048,8192] + scratch KV [16,8,8,128] bf16",
    "gqa_f16": "GQA decode in f16: B32 T1 Hq32 Hkv8 D128 P16 ctx U[512,8192] f16 q/K/V/out",
    "gqa_d64": "GQA decode, head dim 64: B32 T1 Hq32 Hkv8 D64 P16 ctx U[512,8192] bf16",
    "gqa_d256": "GQA decode, head dim 256: B32 T1 Hq32 Hkv8 D256 P16 ctx U[512,8192] bf16",
    "tidar_causal": "TiDAR draft-block decode with a causal draft: B16 T8 Hq32 Hkv8 D128 P16 ctx U[2048,8192] "
                    "+ scratch KV [16,8,8,128] bf16, draft token t sees scratch tokens <= t",
    "tidar_long": "TiDAR 16-token draft in blocks of 4: B16 T16 Hq32 Hkv8 D128 P16 ctx U[2048,8192] "
                  "+ scratch KV [16,16,8,128] bf16 (64 query rows per kv head)",
    "append": "KV-cache append of a 512-token chunk: B64 T512 Hkv8 D128 P16 ctx U[0,4096] bf16",
    "append_fp8": "KV-cache append with e4m3fn quantisation: B64 T512 Hkv2 D256 P16 ctx U[0,8192] "
                  "bf16 rows -> e4m3fn + fp32 per-token scale",
    "append_step": "KV-cache append of one decode step: B32 T1 Hkv8 D128 P16 ctx U[512,8192] bf16",
}
APPEND_CONFIGS = ("append", "append_fp8", "append_step")
APPEND_METRIC = "KV-cache append µs/call and achieved HBM GB/s (fraction of 8 TB/s) on 1 GB300"
# Sources of each decode kernel: its device code, the file that builds its
# instances, and the host code that picks the instance, unit geometry and
# launch plan for a shape (a change to any of them can change its traffic).
SPLIT_KERNEL_SOURCES = ["pa_kernels.cuh", "pa_ptx.cuh", "pa_inst_bf16.cu", "pa_inst_f16.cu", "pa_inst_fp8.cu",
                        "pa_api.cu"]
UMMA_KERNEL_SOURCES = ["pa_umma.cuh", "pa_tc.cuh", "pa_kernels.cuh", "pa_ptx.cuh", "pa_inst_umma.cu",
                       "pa_inst_umma_fp8.cu", "pa_api.cu"]
QROW_KERNEL_SOURCES = ["pa_qrow.cuh", "pa_tc.cuh", "pa_kernels.cuh", "pa_ptx.cuh", "pa_inst_qrow.cu", "pa_api.cu"]
PAIR_KERNEL_SOURCES = ["pa_pair.cuh", "pa_kernels.cuh", "pa_ptx.cuh", "pa_inst_pair.cu", "pa_api.cu"]
KERNEL_NAMES = {1: "pa_split_kernel", 2: "pa_umma_kernel", 3: "pa_qrow_kernel", 4: "pa_pair_kernel"}
KERNEL_SOURCES = {"pa_split_kernel": SPLIT_KERNEL_SOURCES, "pa_umma_kernel": UMMA_KERNEL_SOURCES,
                  "pa_qrow_kernel": QROW_KERNEL_SOURCES, "pa_pair_kernel": PAIR_KERNEL_SOURCES}
APPEND_KERNEL_SOURCES = ["pa_append.cu", "pa_ptx.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


# --------------------------------------------------------------------------- bytes
def algorithmic_bytes(inp) -> int:
    """Bytes a decode call must move at minimum: KV rows of the valid tokens,
    their fp8 scales, the block-table entries in use, q, out, lse,
    context_lens and the draft-block scratch. Split-K partials excluded."""
    s = inp.spec
    lens = inp.context_lens.to(torch.int64)
    tokens = int(lens.sum())
    pages = int(((lens + s.page_size - 1) // s.page_size).sum())
    kv_elem = 1 if s.kv_format == "fp8" else 2
    nbytes = 2 * tokens * s.num_kv_heads * s.head_dim * kv_elem
    if s.kv_format == "fp8":
        nbytes += 2 * tokens * s.num_kv_heads * 4
    nbytes += pages * 4
    rows = s.batch * s.q_tokens * s.num_q_heads
    nbytes += rows * s.head_dim * 2 * 2 + rows * 4 + s.batch * 4
    if s.draft_scratch:
        nbytes += 2 * s.batch * s.q_tokens * s.num_kv_heads * s.head_dim * 2
    return nbytes


def append_bytes(inp) -> int:
    """Bytes an append call must move: read the new K and V rows (bf16), write
    them into the cache (bf16, or e4m3fn codes + an fp32 scale per row),
    read context_lens and the block-table entries the new positions use."""
    s = inp.spec
    cap = inp.block_tables.shape[1] * s.page_size
    lens = inp.context_lens.to(torch.int64).clamp(0, cap)
    ends = (lens + s.new_tokens).clamp(max=cap)
    rows = int((ends - lens).sum()) * s.num_kv_heads * 2  # (token, kv head) rows of K and V
    written = s.head_dim + 4 if s.kv_format == "fp8" else 2 * s.head_dim
    pages = int(((ends - 1) // s.page_size - lens // s.page_size + 1).clamp(min=0)[ends > lens].sum())
    return rows * (2 * s.head_dim + written) + pages * 4 + s.batch * 4


def unit_bytes(spec, ctx: int) -> int:
    """Algorithmic bytes of one (sequence, kv head) unit with ctx keys."""
    kv_elem = 1 if spec.kv_format == "fp8" else 2
    n = 2 * ctx * spec.head_dim * kv_elem + (2 * ctx * 4 if spec.kv_format == "fp8" else 0)
    rows = spec.group * spec.q_tokens
    n += rows * spec.head_dim * 2 * 2 + rows * 4 + ((ctx + spec.page_size - 1) // spec.page_size) * 4
    if spec.draft_scratch:
        n += 2 * spec.q_tokens * spec.head_dim * 2
    return n


# --------------------------------------------------------------------------- peaks
def load_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "of measured"
    except Exception:
        return FALLBACK_HBM_GBS, "of fallback"


def kernel_sha(config: str = DEFAULT_CONFIG, kernel: str = "pa_split_kernel") -> str:
    """Hash of the sources of the kernel a workload's roofline is about."""
    h = hashlib.sha256()
    srcs = APPEND_KERNEL_SOURCES if config in APPEND_CONFIGS else KERNEL_SOURCES[kernel]
    for name in srcs:
        with open(os.path.join(ROOT, "paged_kv_attention_15_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic(config: str, kernel: str = "pa_split_kernel"):
    """DRAM bytes per launch of the workload's kernel from the committed ncu
    summary, if it was taken on the current source of that kernel; else
    None."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f).get(config)
        if rec and rec.get("kernel", "pa_split_kernel") == kernel and rec.get("kernel_sha") == kernel_sha(config, kernel):
            return int(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# --------------------------------------------------------------------------- clocks
_REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
            0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
            0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}


class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML (read only)
    every few milliseconds on a background thread."""

    def __init__(self, device_index: int = 0, period_s: float = 0.002):
        self.period = period_s
        self.samples = []
        self.reasons = 0
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self.nvml = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            handle = ctypes.c_void_p()
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            if nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(handle)) != 0:
                if nv.nvmlDeviceGetHandleByIndex_v2(device_index, ctypes.byref(handle)) != 0:
                    return
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
            self.nvml, self.handle = nv, handle
            fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self._reasons_fn = fn
        except Exception:
            self.nvml = None

    def _run(self):
        mhz = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(mhz)) == 0:
                self.samples.append(int(mhz.value))
            if self._reasons_fn(self.handle, ctypes.byref(rs)) == 0:
                self.reasons |= int(rs.value)
            time.sleep(self.period)

    def start(self):
        if self.nvml is not None:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()

    def summary(self):
        if self.nvml is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"], "samples": 0}
        names = [n for bit, n in _REASONS.items() if self.reasons & bit and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": names, "samples": len(self.samples)}


def merge_clocks(timed: dict, kernel_pass: dict) -> dict:
    """Clock record of the timed replays together with the kernel-only pass
    that follows it (the GPU is busy in both)."""
    out = dict(timed)
    out["kernel_pass"] = kernel_pass
    mhz = [x for x in (timed.get("sm_mhz"), kernel_pass.get("sm_mhz")) if x]
    out["samples"] = (timed.get("samples") or 0) + (kernel_pass.get("samples") or 0)
    out["reasons"] = sorted(set(timed.get("reasons") or []) | set(kernel_pass.get("reasons") or []))
    if not timed.get("sm_mhz") and mhz:
        out["sm_mhz"] = mhz[0]
    return out


# --------------------------------------------------------------------------- ranks
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate_throughput(bytes_per_step: int, steps: int, max_elapsed_s: float, world: int) -> float:
    """Whole-job GB/s: every rank ran `steps` steps of `bytes_per_step`."""
    return world * bytes_per_step * steps / max_elapsed_s / 1e9


# --------------------------------------------------------------------------- oracle timing
def _oracle_bits(inp):
    import oracle

    oi = oracle.as_oracle_inputs(inp.numpy_bits(), inp.spec.kv_format)
    if inp.spec.draft_block is not None:
        oi["draft_block"] = inp.spec.draft_block
    return oi


def _unit_rows(spec, b, g):
    return [(b, t, h) for t in range(spec.q_tokens) for h in range(g * spec.group, (g + 1) * spec.group)]


def oracle_seconds_per_key(inp) -> float:
    """Oracle time per key of one (sequence, kv head) unit, from a prefix of
    up to 4096 keys of the first unit."""
    import oracle

    spec = inp.spec
    bits = _oracle_bits(inp)
    trial = dict(bits)
    trial["context_lens"] = bits["context_lens"].copy()
    probe = int(min(int(trial["context_lens"][0]), 4096))
    trial["context_lens"][0] = max(probe, 1)
    t = time.perf_counter()
    oracle.decode(trial, spec.scale, rows=_unit_rows(spec, 0, 0))
    return max((time.perf_counter() - t) / max(probe, 1), 1e-9)


def oracle_units_run(spec, bits, units, budget_s: float, per_key: float):
    """Runs the oracle, as it stands, on the (sequence, kv head) units in
    order until the budget is spent (whole units; a context prefix of the
    first unit when it alone exceeds the budget). Returns (seconds,
    algorithmic bytes, units done, prefix keys or None)."""
    import oracle

    ctx = bits["context_lens"].astype(np.int64)
    done_s, done_bytes, n_units, prefix = 0.0, 0, 0, None
    for (b, g) in units:
        if done_s >= budget_s:
            break
        c = int(ctx[b])
        run = dict(bits)
        if per_key * c > budget_s - done_s and n_units == 0:
            c = max(1, int((budget_s - done_s) / per_key))
            run["context_lens"] = bits["context_lens"].copy()
            run["context_lens"][b] = c
            prefix = c
        elif per_key * c > 2 * (budget_s - done_s) and n_units > 0:
            break
        t = time.perf_counter()
        oracle.decode(run, spec.scale, rows=_unit_rows(spec, b, g))
        done_s += time.perf_counter() - t
        done_bytes += unit_bytes(spec, c)
        n_units += 1
    return done_s, done_bytes, n_units, prefix


def _all_units(spec, start_unit: int):
    units = [(b, g) for b in range(spec.batch) for g in range(spec.num_kv_heads)]
    k = start_unit % len(units)
    return units[k:] + units[:k]


def oracle_sample_run(inp, budget_s: float, start_unit: int = 0, per_key: float = None):
    """The oracle on one core: whole (sequence, kv head) units from
    start_unit on until the budget is spent. Returns (seconds, algorithmic
    bytes, description)."""
    spec = inp.spec
    if per_key is None:
        per_key = oracle_seconds_per_key(inp)
    secs, nbytes, n_units, prefix = oracle_units_run(spec, _oracle_bits(inp), _all_units(spec, start_unit),
                                                     budget_s, per_key)
    desc = f"{n_units} (sequence, kv head) unit(s) of the {spec.name} workload"
    if prefix is not None:
        desc += f", the first one cut to its first {prefix} keys"
    return secs, nbytes, desc


# The oracle on all host cores: one single-threaded process per core
# (spawned, so safe next to CUDA), the workload's arrays shared with them
# through shared memory (attached, not copied).
_POOL_STATE = {}


def _pool_init(meta, spec):
    from multiprocessing import shared_memory

    # (spawned children share the parent's resource tracker; the parent
    # unlinks the blocks when the pool closes)
    arrays, keep = {}, []
    for name, (shm_name, shape, dtype) in meta["arrays"].items():
        shm = shared_memory.SharedMemory(name=shm_name)
        keep.append(shm)
        arrays[name] = np.ndarray(shape, dtype=np.dtype(dtype), buffer=shm.buf)
    arrays.update(meta["scalars"])
    _POOL_STATE.update(bits=arrays, spec=spec, keep=keep)


def _pool_task(units, budget_s, per_key):
    st = _POOL_STATE
    return oracle_units_run(st["spec"], st["bits"], units, budget_s, per_key)


def _pool_ready(_):
    return os.getpid()


class OraclePool:
    """A pool of `workers` spawned processes running the oracle on disjoint
    units of one workload at once; run() returns the wall time of the whole
    sample, so value = bytes / wall is the throughput of all cores."""

    def __init__(self, inp, workers: int):
        import concurrent.futures
        import multiprocessing as mp
        from multiprocessing import shared_memory

        self.spec = inp.spec
        self.workers = max(1, int(workers))
        bits = _oracle_bits(inp)
        self._shms, meta = [], {"arrays": {}, "scalars": {}}
        for name, v in bits.items():
            if isinstance(v, np.ndarray) and v.nbytes > 0:
                shm = shared_memory.SharedMemory(create=True, size=v.nbytes)
                np.ndarray(v.shape, dtype=v.dtype, buffer=shm.buf)[...] = v
                self._shms.append(shm)
                meta["arrays"][name] = (shm.name, v.shape, v.dtype.str)
            else:
                meta["scalars"][name] = v
        self._ex = None
        try:
            self._ex = concurrent.futures.ProcessPoolExecutor(
                max_workers=self.workers, mp_context=mp.get_context("spawn"), initializer=_pool_init,
                initargs=(meta, self.spec))
            # every worker started and attached before anything is timed
            list(self._ex.map(_pool_ready, range(4 * self.workers)))
        except BaseException:
            self.close()
            raise

    def run(self, budget_s: float, per_key: float, start_unit: int = 0):
        units = _all_units(self.spec, start_unit)
        W = self.workers
        shares = [units[w::W] for w in range(W)]
        t = time.perf_counter()
        res = list(self._ex.map(_pool_task, shares, [budget_s] * W, [per_key] * W))
        wall = time.perf_counter() - t
        nbytes = sum(r[1] for r in res)
        n_units = sum(r[2] for r in res)
        cut = sum(1 for r in res if r[3] is not None)
        desc = (f"{n_units} (sequence, kv head) unit(s) of the {self.spec.name} workload over {W} processes"
                + (f", {cut} of them a context prefix" if cut else ""))
        return wall, nbytes, desc

    def close(self):
        if self._ex is not None:
            self._ex.shutdown(wait=True)
            self._ex = None
        for shm in self._shms:
            shm.close()
            shm.unlink()
        self._shms = []


def cpu_baseline(inp, budget_s: float, workers: int = 0):
    """The oracle timed on one core and on all host cores (os.cpu_count()
    processes, or `workers`). The all-cores run is the reported value."""
    per_key = oracle_seconds_per_key(inp)
    s1, b1, d1 = oracle_sample_run(inp, budget_s, per_key=per_key)
    W = workers or os.cpu_count() or 1
    pool = OraclePool(inp, W)
    try:
        wall, bw, dw = pool.run(budget_s, per_key)
    finally:
        pool.close()
    return {"value": bw / wall / 1e9, "unit": UNIT, "cores": W, "nproc": os.cpu_count(), "kind": "oracle",
            "sample": dw, "seconds": wall,
            "one_core": {"value": b1 / s1 / 1e9, "unit": UNIT, "cores": 1, "sample": d1, "seconds": s1},
            "threads_per_process": 1}


# --------------------------------------------------------------------------- arms
def workload_spec(args):
    """The workload's spec; --batch shrinks it (profiling captures only)."""
    spec = gen.SPECS[args.config]
    if args.batch:
        lens = spec.context_lens[: args.batch] if spec.context_lens is not None else None
        spec = dataclasses.replace(spec, batch=args.batch, context_lens=lens)
    return spec


def run_ours(args, world, rank, local):
    from paged_kv_attention_15_gb300 import binding as pb

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    spec = workload_spec(args)
    host = gen.make_inputs(spec)
    pb.lib()
    pb.set_kernel_path({"auto": pb.KERNEL_AUTO, "warp": pb.KERNEL_WARP_MMA, "tcgen05": pb.KERNEL_TCGEN05,
                        "tcgen05-qrow": pb.KERNEL_TCGEN05_QROW, "warp-pair": pb.KERNEL_WARP_PAIR}[args.kernel_path])
    sets = [host.to(dev), host.to(dev)]  # alternated: each step reads KV not in L2
    kname = KERNEL_NAMES[pb.kernel_for_inputs(sets[0])]
    shape = pb.make_shape(sets[0].q, sets[0].k_cache, sets[0].block_tables)
    ws_bytes = pb.workspace_size(shape, args.num_splits)
    wss = [torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev) for _ in sets]
    outs = [torch.empty_like(s.q) for s in sets]
    lses = [torch.empty(s.q.shape[:3], dtype=torch.float32, device=dev) for s in sets]
    stream = torch.cuda.current_stream(dev)

    def step(i):
        j = i & 1
        pb.decode_inputs(sets[j], out=outs[j], lse=lses[j], workspace=wss[j], num_splits=args.num_splits,
                         stream=stream)

    nbytes = algorithmic_bytes(host)
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    assert pb.device_error() == 0

    # One CUDA graph per input set (the first call on a device already ran
    # outside capture); steps replay them alternately.
    graphs = []
    cap_stream = torch.cuda.Stream(dev)
    cap_stream.wait_stream(stream)
    with torch.cuda.stream(cap_stream):
        for j in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap_stream):
                pb.decode_inputs(sets[j], out=outs[j], lse=lses[j], workspace=wss[j], num_splits=args.num_splits)
            graphs.append(g)
    torch.cuda.synchronize(dev)
    # Not an empty graph: a replay rewrites the output, NaN-filled first
    # (every output row is written, zeros for a sequence with no keys).
    for j in range(2):
        outs[j].fill_(float("nan"))
    with torch.cuda.stream(cap_stream):
        for j in range(2):
            graphs[j].replay()
    torch.cuda.synchronize(dev)
    for j in range(2):
        if not bool(torch.isfinite(outs[j]).all()):
            raise RuntimeError("a captured decode graph did not write its output")
    with torch.cuda.stream(cap_stream):
        for i in range(args.warmup):
            graphs[i & 1].replay()
    torch.cuda.synchronize(dev)

    # ---- timed region: K graph replays = K decode calls
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    with torch.cuda.stream(cap_stream):
        t0.record(cap_stream)
        for i in range(args.steps):
            graphs[i & 1].replay()
        t1.record(cap_stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks.stop()
    elapsed_ms = t0.elapsed_time(t1)
    assert pb.device_error() == 0

    # ---- the split kernel alone: CUDA events around its launch (eager calls),
    # at least --kernel-steps calls whatever --steps is, clocks sampled
    # across them as well
    kcalls = max(1, args.kernel_steps)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(kcalls)]
    for a, b in ev:  # torch creates the CUDA event handles on first record
        a.record(stream)
        b.record(stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    kclocks = ClockSampler(local)
    kclocks.start()
    e0.record(stream)
    for i in range(kcalls):
        pb.arm_profile_events(ev[i][0], ev[i][1])
        step(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    kclocks.stop()
    assert pb.device_error() == 0
    split_ms = [a.elapsed_time(b) for a, b in ev]
    eager_ms_per_call = e0.elapsed_time(e1) / kcalls

    max_ms = max_over_ranks(elapsed_ms, world, dev)
    ms_per_step = max_ms / args.steps
    value = aggregate_throughput(nbytes, args.steps, max_ms / 1e3, world)
    split_mean_ms = sum(split_ms) / len(split_ms)
    split_median_ms = statistics.median(split_ms)
    peak, peak_src = load_peak()
    achieved = nbytes / (split_median_ms / 1e3) / 1e9

    e2e = run_e2e(args, host, dev, pb, nbytes, world)
    serving = run_serving_step(args, host, dev, pb, nbytes, world)

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": spec.kv_format, "data": "synthetic",
        "config": {
            "workload": WORKLOADS[args.config] + (f" (batch cut to {spec.batch})" if args.batch else ""),
            "batch": spec.batch, "q_tokens": spec.q_tokens,
            "num_q_heads": spec.num_q_heads, "num_kv_heads": spec.num_kv_heads, "head_dim": spec.head_dim,
            "page_size": spec.page_size, "num_splits": args.num_splits, "seed": spec.seed,
            "split_kernel": kname, "kernel_path": args.kernel_path,
            "algorithmic_bytes_per_step": nbytes,
            "l2": f"inputs larger than L2: two device copies of {nbytes / 1e6:.0f} MB alternated",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "us_per_call": ms_per_step * 1e3,
        "frac_of_8tbs": value / world / NOMINAL_HBM_GBS,
        "kernels_us": {"split": split_median_ms * 1e3, "split_mean": split_mean_ms * 1e3,
                       "split_calls": kcalls, "reduce_and_gaps": (ms_per_step - split_median_ms) * 1e3,
                       "eager_call": eager_ms_per_call * 1e3},
        "timing": "CUDA-graph replays (one graph per input set, alternated); split kernel: median of CUDA-event "
                  f"durations around its launch over {kcalls} eager calls (input sets alternated)",
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": load_traffic(args.config, kname), "peak_source": peak_src,
                     "kernel": kname},
        "clocks": merge_clocks(clocks.summary(), kclocks.summary()),
        "e2e": e2e,
        "e2e_serving_step": serving,
        "gpu_launches": 2 * args.steps if (args.num_splits != 1) else args.steps,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(host, args.cpu_budget, args.cpu_workers)
    return result


def append_oracle_run(host, budget_s: float, start_seq: int = 0):
    """The append oracle, as it stands, on whole sequences until the budget
    is spent. Returns (seconds, algorithmic bytes, description)."""
    from oracle import kv_append as ka

    bits = host.numpy_bits()
    names = [n for n in ("k_cache", "v_cache", "k_scale", "v_scale") if n in bits]
    spec = host.spec
    done_s, done_b, n = 0.0, 0, 0
    per_seq = append_bytes(host) / spec.batch
    while done_s < budget_s and n < spec.batch:
        b = (start_seq + n) % spec.batch
        # The oracle returns copies of the caches it is given: give it the
        # sequence's own pages (block table renumbered), not the whole pool.
        row = bits["block_tables"][b:b + 1]
        pages = row[row >= 0]
        caches = {nm: bits[nm][pages] for nm in names}
        local = np.where(row >= 0, np.cumsum(row >= 0, axis=1) - 1, -1).astype(np.int32)
        t = time.perf_counter()
        ka.append(caches, bits["k_new"][b:b + 1], bits["v_new"][b:b + 1], local, bits["context_lens"][b:b + 1],
                  spec.page_size)
        done_s += time.perf_counter() - t
        done_b += per_seq
        n += 1
    return done_s, int(done_b), f"{n} sequence(s) of the {spec.name} workload (mean bytes per sequence)"


def run_append(args, world, rank, local):
    """One step = one KV-cache append call over the whole batch."""
    from paged_kv_attention_15_gb300 import binding as pb

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    host = gen.make_append_inputs(gen.APPEND_SPECS[args.config])
    spec = host.spec
    pb.lib()
    sets = [host.to(dev), host.to(dev)]
    stream = torch.cuda.current_stream(dev)

    def call(d, st):
        pb.kv_append(d.k_new, d.v_new, d.block_tables, d.context_lens, d.k_cache, d.v_cache,
                     k_scale=d.k_scale, v_scale=d.v_scale, stream=st)

    nbytes = append_bytes(host)
    for i in range(args.warmup):
        call(sets[i & 1], stream)
    torch.cuda.synchronize(dev)
    graphs = []
    cap_stream = torch.cuda.Stream(dev)
    cap_stream.wait_stream(stream)
    with torch.cuda.stream(cap_stream):
        for j in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap_stream):
                call(sets[j], cap_stream)
            graphs.append(g)
    torch.cuda.synchronize(dev)
    # Not an empty graph: a replay writes the new rows into caches cleared first.
    for j in range(2):
        sets[j].k_cache.zero_()
    with torch.cuda.stream(cap_stream):
        for j in range(2):
            graphs[j].replay()
    torch.cuda.synchronize(dev)
    for j in range(2):
        if not bool(sets[j].k_cache.view(torch.uint8).any()):
            raise RuntimeError("a captured append graph did not write the cache")
    with torch.cuda.stream(cap_stream):
        for i in range(args.warmup):
            graphs[i & 1].replay()
    torch.cuda.synchronize(dev)

    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    with torch.cuda.stream(cap_stream):
        t0.record(cap_stream)
        for i in range(args.steps):
            graphs[i & 1].replay()
        t1.record(cap_stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks.stop()
    max_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    ms_per_step = max_ms / args.steps

    # the append kernel alone: CUDA events around eager calls (one launch
    # each), at least --kernel-steps of them, clocks sampled across them
    kcalls = max(1, args.kernel_steps)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(kcalls)]
    torch.cuda.synchronize(dev)
    kclocks = ClockSampler(local)
    kclocks.start()
    for i in range(kcalls):
        ev[i][0].record(stream)
        call(sets[i & 1], stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    kclocks.stop()
    kern_ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    peak, peak_src = load_peak()
    achieved = nbytes / (kern_ms / 1e3) / 1e9

    # end to end: the new rows, tables and lengths copied from pinned host
    # memory every step; the result stays in the device cache (no read-back)
    pinned = {n: getattr(host, n).pin_memory() for n in ("k_new", "v_new", "block_tables", "context_lens")}
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d = sets[0]
    k = max(1, min(args.steps, args.e2e_steps))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for it in range(k + 3):
        if it == 3:
            a.record(stream)
        for n, t in pinned.items():
            getattr(d, n).copy_(t, non_blocking=True)
        call(d, stream)
    b.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(a.elapsed_time(b), world, dev) / k

    result = {
        "metric": APPEND_METRIC, "value": aggregate_throughput(nbytes, args.steps, max_ms / 1e3, world),
        "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16->e4m3fn" if spec.kv_format == "fp8" else "bf16", "data": "synthetic",
        "config": {
            "workload": WORKLOADS[args.config], "batch": spec.batch, "new_tokens": spec.new_tokens,
            "num_kv_heads": spec.num_kv_heads, "head_dim": spec.head_dim, "page_size": spec.page_size,
            "seed": spec.seed, "algorithmic_bytes_per_step": nbytes,
            "l2": f"two device copies of the inputs and caches alternated ({nbytes / 1e6:.0f} MB moved per call)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "us_per_call": ms_per_step * 1e3,
        "frac_of_8tbs": aggregate_throughput(nbytes, args.steps, max_ms / 1e3, world) / world / NOMINAL_HBM_GBS,
        "kernels_us": {"append": kern_ms * 1e3, "append_calls": kcalls},
        "timing": "CUDA-graph replays (one graph per input set, alternated); the append kernel from CUDA "
                  "events around eager calls",
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": load_traffic(args.config), "peak_source": peak_src, "kernel": "pa_kv_append_kernel"},
        "clocks": merge_clocks(clocks.summary(), kclocks.summary()),
        "e2e": {"value": nbytes * world / (e2e_ms / 1e3) / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": 0, "steps": k, "ms_per_step": e2e_ms,
                "note": "the appended rows stay in the device cache; nothing is read back"},
        "gpu_launches": args.steps,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        secs, nb, desc = append_oracle_run(host, args.cpu_budget)
        result["cpu_baseline"] = {"value": nb / secs / 1e9, "unit": UNIT, "cores": 1, "nproc": os.cpu_count(),
                                  "kind": "oracle", "sample": desc, "seconds": secs,
                                  "note": "one core: the append oracle is timed single-threaded"}
    return result


def run_serving_step(args, host, dev, pb, nbytes, world):
    """One serving decode step through the public calls, the KV cache resident
    on the device (filled once, untimed): every step copies q, the new
    token's K/V rows, the block table and the lengths (and the draft scratch)
    from pinned host memory, appends the new rows at position C_b - 1
    (quantising them for an fp8 cache), decodes over C_b tokens and reads out
    and lse back. value = the decode's algorithmic bytes / step time."""
    spec = host.spec
    B, Hkv, D = spec.batch, spec.num_kv_heads, spec.head_dim
    devset = host.to(dev)
    gen_new = torch.Generator().manual_seed(spec.seed + 77)
    dt = torch.float16 if spec.kv_format == "f16" else torch.bfloat16  # (f16 rows into an f16 cache)
    k_new = torch.randn(B, 1, Hkv, D, generator=gen_new).to(dt).pin_memory()
    v_new = torch.randn(B, 1, Hkv, D, generator=gen_new).to(dt).pin_memory()
    per_step = {"q": host.q, "block_tables": host.block_tables, "context_lens": host.context_lens}
    if host.k_scratch is not None:
        per_step.update(k_scratch=host.k_scratch, v_scratch=host.v_scratch)
    pinned = {n: t.pin_memory() for n, t in per_step.items()}
    pos_h = (host.context_lens - 1).clamp(min=0).to(torch.int32).pin_memory()  # append position per sequence
    kn_d, vn_d = torch.empty_like(k_new, device=dev), torch.empty_like(v_new, device=dev)
    pos_d = torch.empty_like(pos_h, device=dev)
    shape = pb.make_shape(devset.q, devset.k_cache, devset.block_tables)
    ws = torch.empty(max(pb.workspace_size(shape, args.num_splits), 1), dtype=torch.uint8, device=dev)
    out = torch.empty_like(devset.q)
    lse = torch.empty(devset.q.shape[:3], dtype=torch.float32, device=dev)
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in list(pinned.values()) + [k_new, v_new, pos_h])
    d2h = out.numel() * out.element_size() + lse.numel() * lse.element_size()
    stream = torch.cuda.current_stream(dev)

    def step(st):
        for name, t in pinned.items():
            getattr(devset, name).copy_(t, non_blocking=True)
        kn_d.copy_(k_new, non_blocking=True)
        vn_d.copy_(v_new, non_blocking=True)
        pos_d.copy_(pos_h, non_blocking=True)
        pb.kv_append(kn_d, vn_d, devset.block_tables, pos_d, devset.k_cache, devset.v_cache,
                     k_scale=devset.k_scale, v_scale=devset.v_scale, stream=st)
        pb.decode_inputs(devset, out=out, lse=lse, workspace=ws, num_splits=args.num_splits, stream=st)
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)

    for _ in range(max(3, min(args.warmup, 10))):
        step(stream)
    torch.cuda.synchronize(dev)
    # The step (copies included) as one CUDA graph, as a serving loop issues it.
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            step(cap)
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize(dev)
    k = max(1, min(args.steps, 200))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    with torch.cuda.stream(cap):
        a.record(cap)
        for _ in range(k):
            g.replay()
        b.record(cap)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(a.elapsed_time(b), world, dev)
    return {"value": aggregate_throughput(nbytes, k, ms / 1e3, world), "unit": UNIT, "us_per_step": ms * 1e3 / k,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": k,
            "kernels": "pa_kv_append(_fp8) + pa_decode*",
            "note": "KV cache resident; the new token's rows appended; each step one CUDA-graph replay of the "
                    "copies, the append, the decode and the read-back"}


def run_e2e(args, host, dev, pb, nbytes, world):
    """Same metric through the public call with host buffers: every step
    copies its inputs from pinned host memory and reads out + lse back."""
    pinned = host.pin_memory()
    devset = host.to(dev)
    shape = pb.make_shape(devset.q, devset.k_cache, devset.block_tables)
    ws = torch.empty(max(pb.workspace_size(shape, args.num_splits), 1), dtype=torch.uint8, device=dev)
    out = torch.empty_like(devset.q)
    lse = torch.empty(devset.q.shape[:3], dtype=torch.float32, device=dev)
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in pinned.tensors().values())
    d2h = out.numel() * out.element_size() + lse.numel() * lse.element_size()
    stream = torch.cuda.current_stream(dev)

    def step():
        for name, t in pinned.tensors().items():
            getattr(devset, name).copy_(t, non_blocking=True)
        pb.decode_inputs(devset, out=out, lse=lse, workspace=ws, num_splits=args.num_splits, stream=stream)
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)

    for _ in range(max(1, min(args.warmup, 3))):
        step()
    torch.cuda.synchronize(dev)
    k = max(1, min(args.steps, args.e2e_steps))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    a.record(stream)
    for _ in range(k):
        step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(a.elapsed_time(b), world, dev)
    return {"value": aggregate_throughput(nbytes, k, ms / 1e3, world), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": k, "ms_per_step": ms / k}


def run_reference_append(args):
    """The append oracle on host cores, each step a bounded sample."""
    host = gen.make_append_inputs(gen.APPEND_SPECS[args.config])
    budget = max(0.002, args.reference_seconds / (args.steps + args.warmup))
    for w in range(args.warmup):
        append_oracle_run(host, budget, start_seq=w)
    secs, nbytes, desc = 0.0, 0, None
    t0 = time.perf_counter()
    for i in range(args.steps):
        s, b, d = append_oracle_run(host, budget, start_seq=args.warmup + i)
        secs += s
        nbytes += b
        desc = desc or d
    wall = time.perf_counter() - t0
    value = nbytes / secs / 1e9
    return {"metric": APPEND_METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": wall * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOADS[args.config]},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"per step: {desc}"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def run_reference(args):
    """The fp64 CPU oracle, as it stands, on host cores: each step is a
    bounded sample of the workload sized so the whole run takes minutes."""
    if args.config in APPEND_CONFIGS:
        return run_reference_append(args)
    spec = workload_spec(args)
    host = gen.make_inputs(spec)
    budget = max(0.002, args.reference_seconds / (args.steps + args.warmup))
    per_key = oracle_seconds_per_key(host)
    W = args.cpu_workers or os.cpu_count() or 1
    pool = OraclePool(host, W)
    try:
        for w in range(args.warmup):
            pool.run(budget, per_key, start_unit=w)
        secs, nbytes, desc = 0.0, 0, None
        for i in range(args.steps):
            s, b, d = pool.run(budget, per_key, start_unit=args.warmup + i)
            secs += s
            nbytes += b
            desc = desc or d
    finally:
        pool.close()
    value = nbytes / secs / 1e9
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": secs * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOADS[args.config], "num_splits": args.num_splits},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": W, "nproc": os.cpu_count(), "kind": "oracle",
                             "threads_per_process": 1, "sample": f"per step: {desc}"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (profiling only)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--kernel-steps", type=int, default=300,
                    help="eager calls timed for the dominant kernel alone (independent of --steps)")
    ap.add_argument("--cpu-workers", type=int, default=0, help="oracle processes for the all-cores run (0: all)")
    ap.add_argument("--kernel-path", default="auto", choices=["auto", "warp", "tcgen05", "tcgen05-qrow", "warp-pair"],
                    help="split kernel: automatic choice, the warp-level MMA kernel, or one of the tcgen05 "
                         "kernels (token-major, query-row-major)")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--reference-seconds", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)))
        return 0
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    result = (run_append if args.config in APPEND_CONFIGS else run_ours)(args, world, rank, local)
    if rank == 0:
        print(json.dumps(result))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
