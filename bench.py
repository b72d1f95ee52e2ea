"""Benchmark: HBM GB/s of the packed varlen causal conv1d on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload long16k]
                    [--impl ours|reference]

One step = one kda_packed_conv1d call over one batch of the workload (the
whole hot path: program map, state read/write, taps, SiLU, rounding, plane
stores).  The default workload is one 16384-token prefill chunk of the
Kimi-K3 KDA Q|K|V projection: dim 4608 = 3 x 1536, bf16 x with row stride
6400, FP32 weights / bias / conv state, SiLU.

value = algorithmic bytes moved by all ranks / timed region (GB/s).  The
algorithmic bytes are x read once + out written once + state lines read and
written + weight and bias (halo re-reads not counted).  Consecutive steps use
different copies of the inputs and outputs (rotating sets whose total is far
above the 129 MB L2), so no step finds its data in L2.

--impl reference times the CPU oracle (plain single-threaded C) on a bounded
sample of the same workload on the host cores, as the reference arm.

Prints one JSON line (rank 0).
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
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "HBM GB/s (read+write) & % of GB300 peak; packed QKV conv 16K x 3x1536 bf16"
UNIT = "GB/s"
PAGE_GBS = 4800.0  # the page's ~4.8 TB/s for its packed kernel at 2K-16K x 3x1536 on GB300
PAGE_WORKLOADS = ("long16k", "varlen")  # the workloads inside that range
FALLBACK_HBM_GBS = 6800.0
KERNEL_SRC = os.path.join(ROOT, "linear_attention_prefill_varlen_gb300", "csrc", "kda_conv.cu")
PROFILES = os.path.join(ROOT, "profiles")
L2_BYTES = 129 * 1024 * 1024


def _workload_name(name: str) -> str:
    if not workloads.valid_name(name):
        raise argparse.ArgumentTypeError(f"unknown workload {name!r}")
    return name


def page_range(b: workloads.Batch) -> bool:
    """The page's ~4.8 TB/s figure is for 2K-16K-token prefill chunks at
    3 x 1536 channels."""
    if b.name in PAGE_WORKLOADS:
        return True
    return (b.name.startswith("prefill") and b.dim == 4608 and b.part_dim == 1536
            and 2048 <= b.tokens <= 16384)


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="long16k", type=_workload_name,
                    help="one of %s, or prefill<T> / decode<N> at any size" %
                         ", ".join(sorted(workloads.WORKLOADS)))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--entry", default="packed", choices=["packed", "update"],
                    help="update: kda_conv1d_update (every sequence must be one token long)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target seconds of oracle work for the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--x-dtype", default="bf16", choices=["bf16", "f16", "f32"],
                    help="storage of x and out (fp16 / fp32 go through kda_packed_conv1d_ex)")
    ap.add_argument("--state-width", type=int, default=3, help="conv state positions K >= 3")
    ap.add_argument("--state-layout", default="dense", choices=["dense", "position_major"],
                    help="position_major: (lines, K, dim) memory viewed as (lines, dim, K)")
    ap.add_argument("--weight-layout", default="channel_major",
                    choices=["channel_major", "tap_major"],
                    help="tap_major: (4, dim) memory viewed as (dim, 4)")
    ap.add_argument("--qk-l2norm", action="store_true",
                    help="the *_l2norm entry points: planes 0 and 1 normalised per 128-channel "
                         "head (eps 1e-6); the cpu_baseline stays the plain conv oracle")
    return ap.parse_args(argv)


def measured_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_sha() -> str:
    """Hash of the kernel source's code: comments dropped and whitespace
    collapsed, so that editing a comment keeps recorded counters valid."""
    with open(KERNEL_SRC) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    src = " ".join(src.split())
    return hashlib.sha256(src.encode()).hexdigest()[:16]


STORAGE_SUFFIX = ""  # e.g. "_f32" or "_k4_state-position_major": set by main()


def profile_path(entry: str, workload: str) -> str:
    kernel = "kda_conv1d_update" if entry == "update" else "kda_packed_conv1d"
    if NORM is not None:
        kernel += "_l2norm"
    return os.path.join(PROFILES, f"{kernel}_{workload}{STORAGE_SUFFIX}.md")


def packed_kernel_name(b: workloads.Batch) -> str:
    """The kernel the timed call launches: the decode update, the looping
    short kernel (at most one token per sequence, bf16/f16/fp32 x with a dense
    fp32 width-3 state and a channel-major weight), or the conv kernel."""
    if ENTRY == "update":
        return "kda_conv1d_update_kernel"
    default_state = (b.conv_states.dtype == np.float32 and b.conv_states.shape[2] == 3
                     and LAYOUT_OPTS["state_layout"] == "dense"
                     and LAYOUT_OPTS["weight_layout"] == "channel_major")
    if b.tokens <= b.num_seqs and default_state:
        return "kda_packed_conv1d_loop_kernel"
    return "kda_packed_conv1d_kernel"


def recorded_traffic(entry: str, workload: str) -> dict:
    """Per-launch DRAM bytes (read + write, and each side) recorded from one
    ncu capture in the committed summary of this kernel on this workload, if
    there is one and it was taken on the current kernel source (its sha line
    matches); otherwise None for each."""
    none = {"traffic": None, "traffic_read": None, "traffic_write": None,
            "traffic_source": None}
    try:
        path = profile_path(entry, workload)
        text = open(path).read()
    except OSError:
        return none
    sha = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", text)
    tr = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    rd = re.search(r"dram_read_bytes_per_launch:\s*([0-9]+)", text)
    wr = re.search(r"dram_write_bytes_per_launch:\s*([0-9]+)", text)
    if not sha or not tr or sha.group(1) != kernel_sha():
        return none
    return {"traffic": int(tr.group(1)),
            "traffic_read": int(rd.group(1)) if rd else None,
            "traffic_write": int(wr.group(1)) if wr else None,
            "traffic_source": ("recorded: dram__bytes_read.sum / dram__bytes_write.sum of one "
                               "ncu launch (caches flushed before it; writes still dirty in L2 "
                               "when it ends are not counted), "
                               + os.path.relpath(path, ROOT))}


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
             "clocks.mem,temperature.gpu,temperature.memory")

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"kda_bench_clocks_gpu{device_index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return self
        # nvidia-smi's start-up (NVML initialisation) slows kernel launches
        # down while it runs: wait for its first sample before going on.
        t_end = time.perf_counter() + 10.0
        while time.perf_counter() < t_end and self.proc.poll() is None:
            try:
                if os.path.getsize(self.path) > 0:
                    break
            except OSError:
                pass
            time.sleep(0.02)
        time.sleep(0.1)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self) -> dict | None:
        if self.proc is None:
            return None
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                extra = [float(p) if p not in ("N/A", "[N/A]") else None for p in parts[9:12]]
                extra += [None] * (3 - len(extra))
                rows.append((float(parts[1]), float(parts[2]), parts[4:9], *extra))
            except ValueError:
                continue
        if not rows:
            return None
        sm_max = max(r[1] for r in rows)
        loaded = [r for r in rows if r[0] >= 0.5 * sm_max] or rows
        names = ["active_mask", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(1, 5) if r[2][i] == "Active"})
        out = {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": sm_max,
               "reasons": reasons, "samples": len(rows)}
        if all(r[3] is not None for r in loaded):
            out["mem_mhz"] = statistics.median(r[3] for r in loaded)
        if all(r[4] is not None for r in loaded):
            out["temp_c_max"] = max(r[4] for r in loaded)
        if all(r[5] is not None for r in loaded):
            out["mem_temp_c_max"] = max(r[5] for r in loaded)
        return out


def dist_env() -> tuple[int, int, int]:
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


class Dist:
    """Barrier and max-over-ranks for N > 1 (one process per GPU)."""

    def __init__(self, world: int, backend: str):
        self.world = world
        self.pg = None
        if world > 1:
            import torch.distributed as dist

            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, v: float, device) -> float:
        if self.pg is None:
            return v
        t = torch.tensor([v], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def aggregate(dist: Dist, world: int, nbytes_per_rank: int, region_ms: float, steps: int,
              device) -> tuple[float, float]:
    """Whole-job figures from one rank's timed region: the slowest rank's time
    per step, and the bytes all ranks moved per second (GB/s)."""
    slowest = dist.max(region_ms, device)
    ms_per_step = slowest / steps
    return ms_per_step, world * nbytes_per_rank / (ms_per_step * 1e-3) / 1e9


LAYOUT_OPTS = {"state_layout": "dense", "weight_layout": "channel_major"}  # set by main()


def x_host_array(b: workloads.Batch, dense_x: bool) -> np.ndarray:
    """x as stored: 16-bit patterns as int16, fp32 as float32."""
    x_np = b.x_buf[:, b.col_offset:b.col_offset + b.dim] if dense_x else b.x_buf
    x_np = np.ascontiguousarray(x_np)
    return x_np if b.x_dtype == "f32" else x_np.view(np.int16)


def out_dtype(b: workloads.Batch):
    return torch.float32 if b.x_dtype == "f32" else torch.int16


def upload(b: workloads.Batch, dev, dense_x: bool = False) -> dict:
    """Device copies of one batch.  dense_x stores x as (tokens, dim) contiguous.
    The conv state and the weight take the memory orders LAYOUT_OPTS names."""
    x = torch.from_numpy(x_host_array(b, dense_x)).to(dev)
    esz = 4 if b.x_dtype == "f32" else 2
    st_np = b.conv_states
    if LAYOUT_OPTS["state_layout"] == "position_major":
        st_np = np.ascontiguousarray(st_np.transpose(0, 2, 1))
    if st_np.dtype == np.uint16:  # bf16 bits
        states = torch.from_numpy(st_np.view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        states = torch.from_numpy(st_np).to(dev)
    if LAYOUT_OPTS["state_layout"] == "position_major":
        states = states.transpose(1, 2)
    if LAYOUT_OPTS["weight_layout"] == "tap_major":
        weight = torch.from_numpy(np.ascontiguousarray(b.weight.T)).to(dev).t()
    else:
        weight = torch.from_numpy(b.weight).to(dev)
    return {
        "x": x,
        "x_ptr": x.data_ptr() + (0 if dense_x else esz * b.col_offset),
        "x_row_stride": b.dim if dense_x else b.row_stride,
        "weight": weight,
        "bias": None if b.bias is None else torch.from_numpy(b.bias).to(dev),
        "conv_states": states,
        "cache_indices": torch.from_numpy(b.cache_indices).to(dev),
        "has_initial_state": torch.from_numpy(b.has_initial_state).to(dev),
        "query_start_loc": torch.from_numpy(b.query_start_loc).to(dev),
        "out": torch.empty((b.dim // b.part_dim, b.tokens, b.part_dim), dtype=out_dtype(b),
                           device=dev),
    }


ENTRY = "packed"


def upload_probe(b: workloads.Batch) -> dict:
    """Host stand-ins with the strides upload() gives, for layout decisions."""
    st = torch.empty(b.conv_states.shape, dtype=torch.bfloat16 if b.conv_states.dtype == np.uint16
                     else torch.float32)
    if LAYOUT_OPTS["state_layout"] == "position_major":
        st = torch.empty((st.shape[0], st.shape[2], st.shape[1]), dtype=st.dtype).transpose(1, 2)
    w = torch.empty(4, b.dim).t() if LAYOUT_OPTS["weight_layout"] == "tap_major" else \
        torch.empty(b.dim, 4)
    return {"conv_states": st, "weight": w}


def state_layout(pkg, b: workloads.Batch, s: dict):
    """None for the default layout (bf16 x, a dense width-3 fp32 state, a
    channel-major weight), else the kda_conv_layout_t of these tensors."""
    st, w = s["conv_states"], s["weight"]
    default = (b.x_dtype == "bf16" and st.dtype == torch.float32 and st.size(2) == 3
               and st.is_contiguous() and tuple(w.stride()) == (4, 1))
    if default:
        return None
    dt = {"bf16": pkg.KDA_DTYPE_BF16, "f16": pkg.KDA_DTYPE_F16, "f32": pkg.KDA_DTYPE_F32}
    sdt = pkg.KDA_DTYPE_BF16 if st.dtype == torch.bfloat16 else pkg.KDA_DTYPE_F32
    return pkg.make_layout(dt[b.x_dtype], st.size(2), st.stride(), w.stride(), sdt)


NORM = None  # --qk-l2norm: planes 0 and 1 normalised per 128-channel head


def call(pkg, b: workloads.Batch, s: dict, stream) -> None:
    if "layout" not in s:
        s["layout"] = state_layout(pkg, b, s)
    if NORM is not None:
        lay = s["layout"] or pkg.make_layout(pkg.KDA_DTYPE_BF16, 3, (3 * b.dim, 3, 1), (4, 1))
        if ENTRY != "update" and s["layout"] is None:
            lay = None
        if ENTRY == "update":
            pkg.kda_conv1d_update_l2norm(
                s["x_ptr"], s["x_row_stride"], b.tokens, b.dim, b.part_dim, s["weight"],
                s["bias"], s["conv_states"], s["cache_indices"], b.null_block_id, b.activation,
                s["out"], lay, NORM, stream)
        else:
            pkg.kda_packed_conv1d_l2norm(
                s["x_ptr"], s["x_row_stride"], b.tokens, b.dim, b.part_dim, s["weight"],
                s["bias"], s["conv_states"], s["cache_indices"], s["has_initial_state"],
                s["query_start_loc"], b.num_seqs, b.null_block_id, b.activation, s["out"], lay,
                NORM, stream)
        return
    if ENTRY == "update":
        pkg.kda_conv1d_update(s["x_ptr"], s["x_row_stride"], b.tokens, b.dim, b.part_dim,
                              s["weight"], s["bias"], s["conv_states"], s["cache_indices"],
                              b.null_block_id, b.activation, s["out"], s["layout"], stream)
        return
    if s["layout"] is not None:
        pkg.kda_packed_conv1d_ex(s["x_ptr"], s["x_row_stride"], b.tokens, b.dim, b.part_dim,
                                 s["weight"], s["bias"], s["conv_states"], s["cache_indices"],
                                 s["has_initial_state"], s["query_start_loc"], b.num_seqs,
                                 b.null_block_id, b.activation, s["out"], s["layout"], stream)
        return
    pkg.kda_packed_conv1d(s["x_ptr"], s["x_row_stride"], b.tokens, b.dim, b.part_dim,
                          s["weight"], s["bias"], s["conv_states"], s["cache_indices"],
                          s["has_initial_state"], s["query_start_loc"], b.num_seqs,
                          b.null_block_id, b.activation, s["out"], stream)


SETTLE_S = 0.2


def settle(dev, stream, seconds: float = SETTLE_S) -> None:
    """Device copies between two 256 MB scratch buffers for about `seconds`,
    ending right before the warm-up steps, so that the GPU's clocks and power
    state are those of a busy GPU (as between a model's layers) when the
    warm-up and the timed region start.  Outside the timed region; the
    buffers are freed afterwards."""
    a = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)
    c = torch.empty_like(a)
    t_end = time.perf_counter() + seconds
    with torch.cuda.stream(stream):
        while time.perf_counter() < t_end:
            for _ in range(16):
                c.copy_(a)
            stream.synchronize()
    del a, c


def prepare(pkg, b: workloads.Batch, s: dict, stream: int):
    """The C function and argument tuple of the call `call` makes on set s,
    every pointer and struct reference converted beforehand, so that a timed
    step is the C-ABI call alone.  Returns (function, args)."""
    import ctypes

    lib = pkg.lib()
    if "layout" not in s:
        s["layout"] = state_layout(pkg, b, s)

    def ptr(t):
        return None if t is None else t.data_ptr()

    def ref(o):
        return None if o is None else ctypes.byref(o)

    common = (s["x_ptr"], s["x_row_stride"], b.tokens, b.dim, b.part_dim, ptr(s["weight"]),
              ptr(s["bias"]), ptr(s["conv_states"]), ptr(s["cache_indices"]))
    packed_meta = (ptr(s["has_initial_state"]), ptr(s["query_start_loc"]), b.num_seqs)
    lay = s["layout"]
    if NORM is not None:
        if lay is None and ENTRY == "update":
            lay = s["norm_layout"] = pkg.make_layout(pkg.KDA_DTYPE_BF16, 3, (3 * b.dim, 3, 1),
                                                     (4, 1))
        if ENTRY == "update":
            return lib.kda_conv1d_update_l2norm, common + (
                b.null_block_id, b.activation, ptr(s["out"]), ref(lay), ref(NORM), stream)
        return lib.kda_packed_conv1d_l2norm, common + packed_meta + (
            b.null_block_id, b.activation, ptr(s["out"]), ref(lay), ref(NORM), stream)
    if ENTRY == "update":
        return lib.kda_conv1d_update, common + (b.null_block_id, b.activation, ptr(s["out"]),
                                                ref(lay), stream)
    if lay is not None:
        return lib.kda_packed_conv1d_ex, common + packed_meta + (
            b.null_block_id, b.activation, ptr(s["out"]), ref(lay), stream)
    return lib.kda_packed_conv1d, common + packed_meta + (b.null_block_id, b.activation,
                                                          ptr(s["out"]), stream)


def check_statuses(pkg, statuses) -> None:
    bad = [st for st in statuses if st != 0]
    if bad:
        pkg._binding._check(bad[0])


def time_device(pkg, b: workloads.Batch, sets: list, steps: int, warmup: int, dist: Dist,
                dev, flush: torch.Tensor | None = None) -> dict:
    """W untimed steps, then exactly K timed steps between barrier+sync pairs,
    each step on the next input/output set, on one stream.  Before the
    warm-up, `settle` keeps the GPU busy for 0.2 s with device copies.

    Without `flush` the K launches run back to back between two region events
    (as a model's layers would issue them); the average launch duration is the
    region over K.  With `flush` (batches too small to rotate out of L2) a
    buffer larger than L2 is rewritten before each step and each launch is
    bracketed by its own events, which then give the step time.  Afterwards,
    outside the timed region, up to 200 more launches with per-launch events
    give the isolated launch time."""
    stream = torch.cuda.Stream(device=dev)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    starts = [ev() for _ in range(steps)] if flush is not None else []
    ends = [ev() for _ in range(steps)] if flush is not None else []
    region0, region1 = ev(), ev()
    # The clock sampler starts before the warm-up, and the GPU is kept busy
    # from there to the timed region: an idle GPU, or nvidia-smi still
    # starting, slowed a 20-step region down by 2-9 % on GB300.
    with ClockSampler(dev.index or 0) as clocks:
        settle(dev, stream)
        for i in range(warmup):
            call(pkg, b, sets[i % len(sets)], stream.cuda_stream)
        # the rotation continues from the warm-up: no step reuses the set of
        # the step before it; each step is the prepared C-ABI call
        prepared = [prepare(pkg, b, sets[(warmup + i) % len(sets)], stream.cuda_stream)
                    for i in range(steps)]
        statuses = []
        dist.barrier()
        torch.cuda.synchronize(dev)
        region0.record(stream)
        for i, (fn, args) in enumerate(prepared):
            if flush is not None:
                with torch.cuda.stream(stream):
                    flush.fill_(i & 0xFF)
                starts[i].record(stream)
            statuses.append(fn(*args))
            if flush is not None:
                ends[i].record(stream)
        region1.record(stream)
        torch.cuda.synchronize(dev)
        check_statuses(pkg, statuses)
    dist.barrier()
    region_ms = region0.elapsed_time(region1)
    if flush is not None:
        launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        step_ms = sum(launch_ms)
    else:
        step_ms = region_ms
    # isolated launches, for reference (events between launches prevent overlap)
    n_iso = min(200, max(steps, 1))
    iso = [(ev(), ev()) for _ in range(n_iso)]
    for i, (s0, s1) in enumerate(iso):
        if flush is not None:
            with torch.cuda.stream(stream):
                flush.fill_(i & 0xFF)
        s0.record(stream)
        call(pkg, b, sets[(warmup + steps + i) % len(sets)], stream.cuda_stream)
        s1.record(stream)
    torch.cuda.synchronize(dev)
    iso_ms = [s0.elapsed_time(s1) for s0, s1 in iso]
    return {"step_ms_total": step_ms, "region_ms": region_ms, "iso_ms": iso_ms,
            "clocks": clocks.summary()}


def time_graph(pkg, b: workloads.Batch, sets: list, launches: int, dev) -> float:
    """The same launches captured in one CUDA graph (rotating over the sets)
    and replayed: microseconds per launch over one timed replay, after one
    untimed replay.  Outside the timed region of the bench step."""
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        call(pkg, b, sets[0], stream.cuda_stream)  # first use outside capture
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        cur = torch.cuda.current_stream().cuda_stream
        for i in range(launches):
            call(pkg, b, sets[i % len(sets)], cur)
    g.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) * 1e3 / launches


def time_hot(pkg, b: workloads.Batch, sets: list, launches: int, dev) -> float:
    """Hot-L2 figure: the same buffer set every launch, back to back, so that
    whatever of it fits in L2 stays there.  Microseconds per launch; outside
    the timed region of the bench step and reported only as context."""
    stream = torch.cuda.Stream(device=dev)
    for _ in range(20):
        call(pkg, b, sets[0], stream.cuda_stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(launches):
        call(pkg, b, sets[0], stream.cuda_stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) * 1e3 / launches


def time_copy(nbytes: int, launches: int, dev) -> float:
    """Context for the roofline: a plain device copy (torch copy_) moving the
    same number of bytes as one launch (half read, half written), back to
    back over rotating buffers larger than L2 in total.  Microseconds per
    copy; outside the timed region."""
    half = max(nbytes // 4, 1)  # int16 elements per side
    n = min(max(2, -(-4 * L2_BYTES // (4 * half))), launches + 20)  # no pair used twice in a row
    bufs = [(torch.empty(half, dtype=torch.int16, device=dev),
             torch.empty(half, dtype=torch.int16, device=dev)) for _ in range(n)]
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for i in range(20):
            bufs[i % n][1].copy_(bufs[i % n][0])
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(20, 20 + launches):  # continues after the warm-up's pairs
            bufs[i % n][1].copy_(bufs[i % n][0])
        e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) * 1e3 / launches


def time_e2e(pkg, b: workloads.Batch, steps: int, dev) -> dict:
    """The same call with HOST inputs and result.  Every step copies its x
    (the (tokens, dim) slice) and metadata from pinned host memory, runs the
    conv, and copies the output planes back to pinned host memory.  Steps are
    pipelined over three streams and two device buffer sets: step i+1's
    upload and step i-1's download overlap step i's kernel."""
    x_host = torch.from_numpy(x_host_array(b, dense_x=True)).pin_memory()
    meta_host = [torch.from_numpy(a).pin_memory() for a in
                 (b.query_start_loc, b.cache_indices, b.has_initial_state)]
    bufs = [upload(b, dev, dense_x=True) for _ in range(2)]
    # one conv state shared by both sets: consecutive steps carry it along
    for s in bufs[1:]:
        s["conv_states"] = bufs[0]["conv_states"]
    out_host = [torch.empty(bufs[0]["out"].shape, dtype=out_dtype(b)).pin_memory()
                for _ in range(2)]
    up, comp, down = (torch.cuda.Stream(device=dev) for _ in range(3))
    uploaded = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    downloaded = [torch.cuda.Event() for _ in range(2)]
    for e in downloaded:
        e.record(down)

    def step(i):
        k = i % 2
        s = bufs[k]
        up.wait_event(downloaded[k])  # set k's previous output has left the device
        with torch.cuda.stream(up):
            s["x"].copy_(x_host, non_blocking=True)
            for d, h in zip((s["query_start_loc"], s["cache_indices"], s["has_initial_state"]),
                            meta_host):
                d.copy_(h, non_blocking=True)
        uploaded[k].record(up)
        comp.wait_event(uploaded[k])
        call(pkg, b, s, comp.cuda_stream)
        computed[k].record(comp)
        down.wait_event(computed[k])
        with torch.cuda.stream(down):
            out_host[k].copy_(s["out"], non_blocking=True)
        downloaded[k].record(down)

    for i in range(4):
        step(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(up)
    for i in range(steps):
        step(i)
    e1.record(down)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    h2d = x_host.numel() * x_host.element_size() + sum(h.numel() * h.element_size()
                                                       for h in meta_host)
    d2h = out_host[0].numel() * out_host[0].element_size()
    return {"ms": ms, "h2d": h2d, "d2h": d2h}


def oracle_sample(b: workloads.Batch, seconds: float, max_reps: int = 50) -> dict:
    """The CPU oracle, as it stands, on the whole workload batch, repeated
    until about `seconds` of work (single thread)."""
    import oracle

    oracle.load()
    reps, t_total = 0, 0.0
    while reps < max_reps and (reps == 0 or t_total < seconds):
        st = b.conv_states.copy()
        t = time.perf_counter()
        if st.dtype == np.uint16 or b.x_dtype != "bf16" or st.shape[2] != 3:  # general oracle
            dt = {"bf16": oracle.DTYPE_BF16, "f16": oracle.DTYPE_F16, "f32": oracle.DTYPE_F32}
            oracle.packed_conv1d_ex(b.x_buf, dt[b.x_dtype], b.col_offset, b.dim, b.part_dim,
                                    b.weight, b.bias, st, b.cache_indices, b.has_initial_state,
                                    b.query_start_loc, b.null_block_id, b.activation)
        else:
            oracle.packed_conv1d(b.x_buf, b.col_offset, b.dim, b.part_dim, b.weight, b.bias, st,
                                 b.cache_indices, b.has_initial_state, b.query_start_loc,
                                 b.null_block_id, b.activation)
        t_total += time.perf_counter() - t
        reps += 1
    nbytes = workloads.algorithmic_bytes(b)
    return {"value": nbytes * reps / t_total / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{reps} x the whole {b.name} batch ({b.tokens} tokens x {b.dim} "
                      f"channels), single-threaded C, {t_total:.1f} s"}


def oracle_multicore(b: workloads.Batch, seconds: float, max_reps: int = 50) -> dict:
    """The same oracle on every host core: one worker process per channel
    block (oracle/multicore.py), each running the unchanged oracle on its
    block; a round covers the whole batch once."""
    from oracle import multicore

    with multicore.OraclePool(b) as pool:
        pool.run(1)  # first touch of the shared arrays
        reps, t_total = 0, 0.0
        while reps < max_reps and (reps == 0 or t_total < seconds):
            t_total += pool.run(1)
            reps += 1
        cores = len(pool.workers)
    nbytes = workloads.algorithmic_bytes(b)
    return {"value": nbytes * reps / t_total / 1e9, "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "sample": f"{reps} x the whole {b.name} batch ({b.tokens} tokens x {b.dim} "
                      f"channels), the single-threaded C oracle run on {cores} channel blocks "
                      f"in {cores} processes at once, {t_total:.1f} s"}


def cpu_baseline(b: workloads.Batch, seconds: float) -> dict:
    """The oracle on all host cores, with the single-threaded run beside it."""
    single = oracle_sample(b, seconds / 2)
    multi = oracle_multicore(b, seconds / 2)
    multi["single_thread"] = {"value": single["value"], "cores": 1, "sample": single["sample"]}
    return multi


def sample_rows(b: workloads.Batch, rows: int) -> workloads.Batch:
    """The first `rows` token rows of a batch as its own call (sequences cut there)."""
    c = b.copy()
    c.x_buf = np.ascontiguousarray(b.x_buf[:rows])
    qsl = np.minimum(b.query_start_loc, rows).astype(np.int32)
    c.query_start_loc = qsl
    return c


def base_line(args, world: int, value: float, ms: float, b: workloads.Batch, extra: dict) -> dict:
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 6),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {
            "workload": b.name, "tokens": b.tokens, "num_seqs": b.num_seqs, "dim": b.dim,
            "part_dim": b.part_dim, "x_row_stride": b.row_stride,
            "activation": "silu" if b.activation else "none", "bias": b.bias is not None,
            "storage": (f"x/out {b.x_dtype}, weight/bias fp32, conv_state "
                        + ("bf16" if b.conv_states.dtype == np.uint16 else "fp32")
                        + f" width {b.conv_states.shape[2]}"),
            "layout": dict(LAYOUT_OPTS),
            "bytes_per_step_per_gpu": workloads.algorithmic_bytes(b),
            "parallelism": f"replicas x{world}",
        },
    }
    line.update(extra)
    return line


def make_workload(args) -> workloads.Batch:
    """The named workload, stored as the --x-dtype / --state-width options say
    (the same draws otherwise)."""
    kw = {}
    if args.x_dtype != "bf16":
        kw["x_dtype"] = args.x_dtype
    if args.state_width != 3:
        kw["state_width"] = args.state_width
    return workloads.by_name(args.workload, **kw)


def run_reference(args) -> None:
    rank, world, _ = dist_env()
    if rank != 0:
        return  # the reference arm runs on rank 0 alone
    import oracle
    from oracle import multicore

    oracle.load()
    b = make_workload(args)
    with multicore.OraclePool(b) as pool:  # the whole batch once, to size the sample
        pool.run(1)
        per_row = pool.run(1) / b.tokens
    budget = 45.0 / max(1, args.steps + args.warmup)
    rows = int(max(16, min(b.tokens, budget / max(per_row, 1e-9))))
    s = sample_rows(b, rows)
    with multicore.OraclePool(s) as pool:
        for _ in range(args.warmup):
            pool.run(1)
        secs = sum(pool.run(1) for _ in range(args.steps))
        cores = len(pool.workers)
    nbytes = workloads.algorithmic_bytes(s)
    value = nbytes * args.steps / secs / 1e9
    sample = (f"per step: the first {rows} token rows of the {b.name} batch (all {b.dim} "
              f"channels), the single-threaded C oracle on {cores} channel blocks in "
              f"{cores} processes at once")
    line = base_line(args, world, value, secs * 1e3 / args.steps, b, {
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    })
    line["config"]["bytes_per_step_per_gpu"] = nbytes
    line["config"]["sample_rows"] = rows
    print(json.dumps(line), flush=True)


def run_ours(args) -> None:
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = Dist(world, "nccl")
    import linear_attention_prefill_varlen_gb300 as pkg

    pkg.lib()
    b = make_workload(args)
    if ENTRY == "update" and not (np.diff(b.query_start_loc) == 1).all():
        raise SystemExit("--entry update needs a batch of one-token sequences (e.g. --workload decode)")
    nbytes = workloads.algorithmic_bytes(b)
    out_bytes = (b.dim // b.part_dim) * b.tokens * b.part_dim * (4 if b.x_dtype == "f32" else 2)
    footprint = b.x_buf.nbytes + out_bytes + b.conv_states.nbytes
    n_sets = min(max(3, -(-4 * L2_BYTES // footprint)), 16)
    sets = [upload(b, dev) for _ in range(n_sets)]
    flush = None
    if n_sets * footprint < 4 * L2_BYTES:  # too small to rotate out of L2: flush instead
        flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize(dev)

    t = time_device(pkg, b, sets, args.steps, args.warmup, dist, dev, flush)
    ms_per_step, value = aggregate(dist, world, nbytes, t["step_ms_total"], args.steps, dev)
    iso_median = dist.max(statistics.median(t["iso_ms"]), dev)
    graph_us = None
    if flush is None:  # back-to-back timing only: a flush cannot live inside the graph
        graph_us = dist.max(time_graph(pkg, b, sets, min(args.steps, 500), dev), dev)
    iso_min = dist.max(min(t["iso_ms"]), dev)
    hot_us = dist.max(time_hot(pkg, b, sets, min(max(args.steps, 1), 500), dev), dev)
    copy_us = dist.max(time_copy(nbytes, min(max(args.steps, 1), 500), dev), dev)

    e2e = time_e2e(pkg, b, args.e2e_steps, dev)
    e2e_ms = dist.max(e2e["ms"], dev)
    del sets
    dist.close()
    if rank != 0:
        return

    peak, peak_kind = measured_peaks()
    achieved = nbytes / (ms_per_step * 1e-3) / 1e9
    extra = {
        "vs_baseline": (round(value / world / PAGE_GBS, 4)
                        if ENTRY == "packed" and NORM is None and page_range(b)
                        else None),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     **recorded_traffic(ENTRY, b.name), "peak_source": peak_kind,
                     "kernel": packed_kernel_name(b),
                     "launch_us_mean": round(ms_per_step * 1e3, 3),
                     "launch_us_isolated_median": round(iso_median * 1e3, 3),
                     "launch_us_isolated_min": round(iso_min * 1e3, 3),
                     "launch_us_graph_replay": None if graph_us is None else round(graph_us, 3),
                     "launch_us_hot_l2": round(hot_us, 3),
                     "copy_us_same_bytes": round(copy_us, 3),
                     "copy_same_bytes": ("torch copy_ of the launch's algorithmic bytes (half "
                                         "read, half written), back to back over rotating "
                                         "buffers; context for frac, not the value"),
                     "hot_l2": (f"one buffer set of {footprint / 1e6:.0f} MB every launch, back "
                                f"to back ({'inside' if footprint <= L2_BYTES else 'larger than'}"
                                f" the 129 MB L2); context only, not the value"),
                     "timing": ("back-to-back launches, region events / K" if flush is None else
                                "per-launch events after an L2 flush")},
        "e2e": {"value": round(world * nbytes / (e2e_ms * 1e-3) / 1e9, 3), "unit": UNIT,
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": round(e2e_ms, 4),
                "note": ("x staged dense (row stride = dim) from pinned host memory; steps "
                         "pipelined over upload / compute / download streams")},
        "gpu_launches": args.steps,
        "clocks": t["clocks"],
        "tokens_per_s": round(world * b.tokens / (ms_per_step * 1e-3), 1),
    }
    line = base_line(args, world, value, ms_per_step, b, extra)
    if flush is None:
        line["config"]["l2"] = (f"{n_sets} rotating input/output/state sets of "
                                f"{footprint / 1e6:.0f} MB (> 129 MB L2 in total); no step reuses "
                                f"the previous step's buffers")
    else:
        line["config"]["l2"] = ("a 512 MB buffer rewritten before every step (L2 flush, outside "
                                "the per-launch events); value from the launches' own time")
    line["config"]["settle"] = (f"{SETTLE_S} s of device copies right before the warm-up "
                                f"steps (clocks and power state of a busy GPU); outside the "
                                f"timed region")
    line["config"]["kernel_source_sha"] = kernel_sha()
    line["config"]["entry"] = "kda_conv1d_update" if ENTRY == "update" else "kda_packed_conv1d"
    if ENTRY != "update" and NORM is None and state_layout(pkg, b, upload_probe(b)) is not None:
        line["config"]["entry"] = "kda_packed_conv1d_ex"
    if NORM is not None:
        line["config"]["entry"] += "_l2norm"
        line["config"]["qk_l2norm"] = {"planes": [0, 1], "head_dim": 128, "eps": 1e-6}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(b, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def main(argv=None) -> None:
    global ENTRY, NORM
    args = parse_args(argv)
    ENTRY = args.entry
    LAYOUT_OPTS["state_layout"] = args.state_layout
    LAYOUT_OPTS["weight_layout"] = args.weight_layout
    global STORAGE_SUFFIX
    STORAGE_SUFFIX = "".join([
        f"_{args.x_dtype}" if args.x_dtype != "bf16" else "",
        f"_k{args.state_width}" if args.state_width != 3 else "",
        f"_state-{args.state_layout}" if args.state_layout != "dense" else "",
        f"_weight-{args.weight_layout}" if args.weight_layout != "channel_major" else ""])
    if args.qk_l2norm and args.impl == "ours":
        import linear_attention_prefill_varlen_gb300 as pkg

        NORM = pkg.make_l2norm(0b011, 128, 1e-6)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
