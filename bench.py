#!/usr/bin/env python3
"""Benchmark of the CSA2 decode step over an FP4 global KV cache.

One step = one pass of the whole hot path over one batch.  The default
workload is hier_1m: one sequence of 1,048,576 cached FP4 rows (D = 512, 64
query heads, a 64x128 FP8 indexer, top-2048), a Full layer that scores every
row, selects its top 2048 and keeps the hierarchical pool of 2048 blocks of 8
rows, then 7 Reindex layers that rescore only the pool's 16,384 rows and
select afresh; every layer attends over its selected FP4 rows.  Layers run in
order, as in a model where each layer's query depends on the layer before.
Other workloads (--workload full_64k, chain_128k, ...) run their own chains.

Prints one JSON line.  --impl reference times the CPU oracle instead (on a
bounded sample of the same workload).  Under torchrun each rank runs its own
copy of the workload (independent sequences: weak scaling, no collective on
the data path).
"""
import argparse
import json
import re
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tokens/s and achieved HBM GB/s (% of ~8 TB/s) per CSA2 layer step"
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 126 * 1000 * 1000     # B300 L2
L2_FLUSH_BYTES = 256 << 20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="hier_1m")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


# ---------------------------------------------------------------------------
# Algorithmic bytes (bytes that must move) per step
# ---------------------------------------------------------------------------

def step_bytes(wl):
    """Indexer keys scanned + selected FP4 rows + queries (+ appended rows)."""
    from fp4_compressed_sparse_append_b300 import workloads as W
    units = wl.B * wl.P
    row = wl.D // 2 + wl.D // 16
    kb = W.key_bytes(wl)                      # stored bytes of one indexer key
    L = wl.length_after_append
    total, index_bytes = 0, 0
    pool_built = False
    for mode in wl.layers:
        q = units * wl.H * wl.D * 2
        if mode != W.REUSE:
            q += units * wl.HI * (wl.DI + 4)
            if mode == W.REINDEX and wl.pool_blocks and pool_built:
                keys = units * wl.pool_blocks * 8 * kb
            else:
                # P positions of a sequence share one scan of the keys
                keys = wl.B * L * kb
            total += keys
            index_bytes = max(index_bytes, keys + units * wl.HI * (wl.DI + 4))
            if mode == W.FULL and wl.pool_blocks:
                pool_built = True
        total += units * min(wl.K, L) * row + q
        if wl.window:
            # the local FP8 rows of each sequence's windows (positions share rows)
            total += wl.B * (wl.window + wl.P - 1) * wl.D
    if wl.n_append:
        # bf16 rows in, FP4 rows and keys out; given keys are read, projected ones are not
        total += wl.B * wl.n_append * (wl.D * 2 + (0 if wl.project else kb) + row + kb)
        if wl.project:
            total += wl.D * wl.DI * 2                 # the projection matrix, once
    return total, index_bytes


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------

class _Nvml:
    """Read-only NVML queries through the driver's libnvidia-ml (ctypes; no
    Python NVML package is needed).  Clock-event reason bits are NVML's."""

    SW_POWER_CAP, HW_SLOWDOWN, SW_THERMAL, HW_THERMAL = 0x4, 0x8, 0x20, 0x40
    CLOCK_SM = 1

    def __init__(self, index):
        import ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML handle")
        self._ct = ctypes

    def clock(self, fn):
        v = self._ct.c_uint()
        if getattr(self.lib, fn)(self.h, self._ct.c_int(self.CLOCK_SM), self._ct.byref(v)) != 0:
            raise RuntimeError(fn + " failed")
        return v.value

    def reasons(self):
        v = self._ct.c_ulonglong()
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        if fn(self.h, self._ct.byref(v)) != 0:
            raise RuntimeError("clock event reasons failed")
        return v.value


class Clocks:
    """Samples the SM clock and the clock-event reasons while the timed region
    runs (read-only queries: NVML through the driver library every couple of
    milliseconds, else nvidia-smi one-shot queries), in a background thread;
    one sample is always taken at start and one at stop."""

    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    QUERY = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, period_s=0.002):
        self.gpu, self.period = gpu_index, period_s
        self.samples, self.reasons, self.max_mhz, self.error = [], set(), None, None
        self._stop, self._thread, self._nvml = None, None, None

    def _sample(self):
        if self._nvml is not None:
            N = self._nvml
            self.samples.append(N.clock("nvmlDeviceGetClockInfo"))
            self.max_mhz = N.clock("nvmlDeviceGetMaxClockInfo")
            bits = N.reasons()
            for name, c in zip(self.REASONS, (N.HW_SLOWDOWN, N.HW_THERMAL, N.SW_THERMAL, N.SW_POWER_CAP)):
                if bits & c:
                    self.reasons.add(name)
            return
        import subprocess
        out = subprocess.run(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                              "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=10).stdout
        parts = [x.strip() for x in out.strip().split(",")]
        self.samples.append(float(parts[0]))
        self.max_mhz = float(parts[1])
        for name, v in zip(self.REASONS, parts[2:6]):
            if v.lower() == "active":
                self.reasons.add(name)

    def _run(self):
        try:
            while not self._stop.wait(self.period):
                self._sample()
        except Exception as e:
            self.error = repr(e)

    def start(self):
        import threading
        try:
            self._nvml = _Nvml(self.gpu)
        except Exception:
            self._nvml = None
            self.period = max(self.period, 0.05)
        try:
            self._sample()
        except Exception as e:
            self.error = repr(e)
        self._stop = threading.Event()
        self._thread = threading.Thread(target=self._run, daemon=True)
        self._thread.start()

    def stop(self):
        self._stop.set()
        self._thread.join()
        try:
            self._sample()
        except Exception as e:
            self.error = self.error or repr(e)
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [self.error or "no samples"]}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples),
                "source": "nvml" if self._nvml else "nvidia-smi"}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

class L2Flush:
    """Evicts the L2 (126 MB) between timed iterations by reading a 256 MiB
    buffer.  A read leaves clean lines behind, so the timed kernels do not pay
    for writing back the flush's own data."""

    def __init__(self, device):
        import torch
        self.buf = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.out = torch.empty((), dtype=torch.float32, device=device)

    def __call__(self):
        import torch
        torch.sum(self.buf, dim=0, out=self.out)


def build_state(wl, seed, device):
    """Untimed setup: the cache (built through csa_quantize_append) and the
    per-layer arguments with their workspaces.  Returns (cache, layers,
    base_len, more_layers); more_layers() builds another set of layer
    arguments over the same cache, with tensors of its own (the e2e leg
    double-buffers its inputs and outputs across steps)."""
    import torch
    from fp4_compressed_sparse_append_b300 import binding as B
    from fp4_compressed_sparse_append_b300 import workloads as W

    cache = B.Cache(wl.B, wl.capacity, wl.D, wl.DI, device=device, key_format=wl.key_format)
    lat = torch.empty((wl.B, wl.L, wl.D), dtype=torch.int16, device=device)
    ik = torch.empty((wl.B, wl.L, W.key_bytes(wl)), dtype=torch.uint8, device=device)
    for b in range(wl.B):
        lat[b], ik[b] = W.cache_rows(wl, seed, b, device=device)
    w_ik = W.ikey_projection(wl, seed, device=device) if wl.project else None
    if wl.project:
        B.csa_quantize_append_project(cache, lat, w_ik)
    else:
        B.csa_quantize_append(cache, lat, ik)
    del lat, ik
    torch.cuda.synchronize()
    app = W.append_rows(wl, seed, device=device) if wl.n_append else None
    swa = B.Swa(W.local_rows(wl, seed, device=device), wl.window) if wl.window else None

    def more_layers(arena: bool = False):
        """Another set of layer arguments.  arena=True: every layer's q, iq and
        w are views into one device buffer and every layer's output into
        another, so that a step's inputs and outputs move in one copy each;
        returns (layers, inputs buffer, outputs buffer)."""
        inputs = [W.layer_inputs(wl, seed, li, device=device) for li in range(len(wl.layers))]
        outs = [None] * len(wl.layers)
        if arena:
            def carve(tensors):
                sizes = [(t.numel() * t.element_size() + 255) // 256 * 256 for t in tensors]
                buf = torch.empty(sum(sizes), dtype=torch.uint8, device=device)
                views, off = [], 0
                for t, n in zip(tensors, sizes):
                    nb = t.numel() * t.element_size()
                    views.append(buf[off:off + nb].view(t.dtype).view(t.shape))
                    off += n
                return buf, views
            flat = [t for inp in inputs for t in (inp["q"], inp["iq"], inp["w"])]
            in_buf, in_views = carve(flat)
            for v, t in zip(in_views, flat):
                v.copy_(t)
            inputs = [dict(q=in_views[3 * li], iq=in_views[3 * li + 1], w=in_views[3 * li + 2])
                      for li in range(len(wl.layers))]
            out_shape = (wl.B, wl.P, wl.H, wl.D)
            out_buf, outs = carve([torch.empty(out_shape, dtype=torch.float32, device=device)
                                   for _ in wl.layers])
        layers, prev, pool = [], None, None
        for li, mode in enumerate(wl.layers):
            inp = inputs[li]
            la = B.LayerArgs(cache, mode, inp["q"], wl.K, wl.scale, iq=inp["iq"], w=inp["w"], out=outs[li],
                             idx=prev if mode == W.REUSE else None,
                             rows_new=app["rows"] if (app and li == 0) else None,
                             ikeys_new=app["ikeys"] if (app and li == 0 and not wl.project) else None,
                             w_ik=w_ik if (app and li == 0) else None,
                             pool_in=pool if mode == W.REINDEX else None, pool_blocks=wl.pool_blocks,
                             make_pool=(mode == W.FULL and wl.pool_blocks > 0 and pool is None), swa=swa)
            if mode != W.REUSE:
                prev = la.idx
            if la.pool_out is not None:
                pool = la.pool_out
            layers.append(la)
        return (layers, in_buf, out_buf) if arena else layers

    layers = more_layers()
    base_len = cache.lengths.clone()
    return cache, layers, base_len, more_layers


def run_step(cache, layers, base_len, wl):
    from fp4_compressed_sparse_append_b300 import binding as B
    for la in layers:
        B.csa_layer_step(cache, la)


def bench_ours(args, wl, rank, world, local_rank):
    import torch
    from fp4_compressed_sparse_append_b300 import binding as B
    from fp4_compressed_sparse_append_b300 import build as BUILD

    if rank == 0 or not os.path.exists(BUILD.LIB):
        BUILD.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    cache, layers, base_len, more_layers = build_state(wl, args.seed, dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    def reset():
        if wl.n_append:
            cache.lengths.copy_(base_len)      # the step appends rows: start each step from the same cache
        flush()                                # L2 flush between timed iterations

    for _ in range(max(3, args.warmup)):
        reset()
        run_step(cache, layers, base_len, wl)
    torch.cuda.synchronize()
    if B.csa_device_status() != 0:
        raise RuntimeError("device status word set during warm-up")

    # The step is captured once as a CUDA graph (the launches of every layer);
    # each timed iteration replays it.  The L2 flush (and, for appending
    # workloads, the reset of the lengths) runs between the timing events.
    launches0 = B.csa_kernel_launches()
    reset()
    step_graph = capture(lambda: run_step(cache, layers, base_len, wl))
    launches_per_step = B.csa_kernel_launches() - launches0
    for _ in range(2):
        reset()
        step_graph.replay()
    torch.cuda.synchronize()

    clocks = Clocks(local_rank)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    for i in range(args.steps):
        reset()
        ev[i][0].record(stream)
        step_graph.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    clock_info = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms, value = aggregate_over_ranks(sum(step_ms), wl.B * wl.P, args.steps, world, dev)
    ms_per_step = total_ms / args.steps
    sbytes, ibytes = step_bytes(wl)
    gbs = sbytes / (ms_per_step / 1e3) / 1e9

    # Stage timings (the dominant kernel for the roofline): each stage alone.
    stages = stage_times(cache, layers, wl, flush, args.steps, stream)
    layer_ms = layer_times(cache, layers, base_len, wl, flush, args.steps, stream)
    # e2e through the public API with host buffers
    e2e = e2e_run(cache, [more_layers(arena=True), more_layers(arena=True)], base_len, wl, args, stream, flush)
    if B.csa_device_status() != 0:
        raise RuntimeError("device status word set during the timed region")
    return dict(value=value, ms_per_step=ms_per_step, gbs=gbs, step_bytes=sbytes, index_bytes=ibytes, layer_ms=layer_ms,
                clocks=clock_info, launches=launches_per_step * args.steps, stages=stages, e2e=e2e,
                step_ms=step_ms)


def aggregate_over_ranks(total_ms, units_per_rank, steps, world, device):
    """The job's time is its slowest rank's (max over ranks); its throughput is
    the units every rank processed over that time (weak scaling: each rank runs
    the same per-GPU workload on its own sequences, with no data exchange)."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.barrier()
        total_ms = float(t.item())
    return total_ms, world * units_per_rank * steps / (total_ms / 1e3)


def capture(fn):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def layer_kinds(wl):
    """The distinct layer kinds of the chain, in order, with how many layers of
    each kind one step runs: [(kind, first layer index, count)].  A kind is the
    mode plus whether it builds or reads the hierarchical pool."""
    from fp4_compressed_sparse_append_b300 import workloads as W
    kinds, seen = [], {}
    pool_built = False
    for li, mode in enumerate(wl.layers):
        if mode == W.FULL:
            kind = "full+pool" if (wl.pool_blocks and not pool_built) else "full"
            pool_built = pool_built or bool(wl.pool_blocks)
        elif mode == W.REINDEX:
            kind = "reindex.pool" if (wl.pool_blocks and pool_built) else "reindex"
        else:
            kind = "reuse"
        if kind in seen:
            kinds[seen[kind]][2] += 1
        else:
            seen[kind] = len(kinds)
            kinds.append([kind, li, 1])
    return [tuple(k) for k in kinds]


def fused_pool_select(wl, pool_in):
    """Whether csa_layer_step scores and selects a Reindex layer over the
    pool in one kernel (the condition csa_pool_topk supports)."""
    return (pool_in is not None and wl.key_format == "e4m3" and wl.HI <= 64 and wl.DI in (32, 64, 128)
            and pool_in.shape[-1] <= 2048 and wl.K <= 16384)


def stage_times(cache, layers, wl, flush, steps, stream):
    """Times the stages of the first layer of each layer kind one at a time,
    each through its own public call, captured as a CUDA graph and replayed
    with the L2 flushed before every replay (CUDA events on the launching
    stream).  Returns {stage: {"ms", "launches", "kind", "stage"}} where
    launches counts the stage's launches per step."""
    import torch
    from fp4_compressed_sparse_append_b300 import binding as B
    from fp4_compressed_sparse_append_b300 import workloads as W

    dev = cache.device

    def timed(fn):
        g = capture(fn)
        ts = []
        for i in range(max(3, min(steps, 100)) + 3):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            if i >= 3:
                ts.append((a, b))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ts)

    out = {}
    for kind, li, count in layer_kinds(wl):
        la = layers[li]
        q, iq, w = la.tensors["q"], la.tensors["iq"], la.tensors["w"]
        pool_in = la.tensors["pool_in"]
        make_pool = la.pool_out is not None
        if la.struct.mode != W.REUSE and fused_pool_select(wl, pool_in):
            # a Reindex layer over the pool: scores and selection in one kernel
            # (the spread form, as csa_layer_step runs it)
            ws_pool = torch.empty(B.pool_topk_workspace_size(cache, wl.P, pool_in.shape[-1]), dtype=torch.uint8,
                                  device=dev)
            idx = B.csa_pool_topk(cache, iq, w, pool_in, wl.K, workspace=ws_pool)
            torch.cuda.synchronize()
            out[kind + ".pool_topk"] = dict(
                ms=timed(lambda: B.csa_pool_topk(cache, iq, w, pool_in, wl.K, idx=idx, workspace=ws_pool)),
                launches=count, kind=kind, stage="pool_topk")
        elif la.struct.mode != W.REUSE:
            nblk = pool_in.shape[-1] if pool_in is not None else 0
            # a Full layer that builds the pool has its scan write the block
            # maxima, from which the pool is selected (as csa_layer_step does)
            bm = B.block_max_buffer(cache, wl.P) if make_pool else None
            scores = B.csa_index_score(cache, iq, w, pool=pool_in, block_max=bm)
            ws_sel = torch.empty(max(16, B.topk_workspace_size(cache, wl.P, wl.K, nblk,
                                                               wl.pool_blocks if make_pool else 0)),
                                 dtype=torch.uint8, device=dev)
            idx, _ = B.csa_topk(cache, scores, wl.K, pool=pool_in, pool_keep=wl.pool_blocks if make_pool else 0,
                                block_max=bm, workspace=ws_sel)
            torch.cuda.synchronize()
            out[kind + ".index_score"] = dict(
                ms=timed(lambda: B.csa_index_score(cache, iq, w, pool=pool_in, scores=scores, block_max=bm)),
                launches=count, kind=kind, stage="index_score")
            out[kind + ".topk"] = dict(
                ms=timed(lambda: B.csa_topk(cache, scores, wl.K, pool=pool_in,
                                            pool_keep=wl.pool_blocks if make_pool else 0, block_max=bm,
                                            workspace=ws_sel)),
                launches=count, kind=kind, stage="topk")
        else:
            idx = la.idx
        swa = la.swa
        ws_att = torch.empty(max(16, B.attend_swa_workspace_size(cache, wl.P, wl.H, wl.K, swa)), dtype=torch.uint8,
                             device=dev)
        o = torch.empty(q.shape, dtype=torch.float32, device=dev)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
        torch.cuda.synchronize()
        out[kind + ".sparse_attend"] = dict(
            ms=timed(lambda: B.csa_sparse_attend_swa(cache, q, idx, wl.scale, swa, workspace=ws_att, out=o,
                                                     lse=lse)),
            launches=count, kind=kind, stage="sparse_attend")
    return out


def layer_times(cache, layers, base_len, wl, flush, steps, stream):
    """Each layer of the step alone (chains: Full, Reindex, Reuse in order),
    captured as its own graph and replayed with L2 flushed before every
    replay; mean device time per layer in ms.  Layers are sequential calls,
    so no layer reads another's keys from L2."""
    import torch
    from fp4_compressed_sparse_append_b300 import binding as B
    out = []
    n = max(3, min(steps, 50))
    for la in layers:
        g = capture(lambda la=la: B.csa_layer_step(cache, la))
        ts = []
        for i in range(n + 2):
            if wl.n_append:
                cache.lengths.copy_(base_len)
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            if i >= 2:
                ts.append((a, b))
        torch.cuda.synchronize()
        out.append(statistics.mean(x.elapsed_time(y) for x, y in ts))
    return out


def e2e_run(cache, sets, base_len, wl, args, stream, flush):
    """Same steps through the public API with pinned host inputs and outputs:
    each step copies every layer's q/iq/w host->device, runs the layers through
    csa_layer_step and copies every layer's output device->host.

    Two sets of layer arguments alternate between steps; each set's inputs
    are views into one device buffer and its outputs into another, so a
    step's inputs go up in one copy and its outputs come down in one.  The
    copies run on two copy streams, ordered by events: the inputs of step s+1
    go up while step s computes, and the outputs of step s come down while
    step s+1 computes.  The layer calls of each set are captured once as a
    CUDA graph (as a serving loop would run them).  The time is that of the
    whole run, from the first input copy to the end of the last output copy,
    over the steps.  When a step moves more bytes than the L2 holds, nothing
    is flushed between steps (the step's own scan evicts it); otherwise the L2
    flush runs before each step's layer calls, inside the timed run."""
    import torch
    layer_sets = [st[0] for st in sets]
    dev_in = [st[1] for st in sets]
    dev_out = [st[2] for st in sets]
    host_in = dev_in[0].cpu().pin_memory()  # both sets hold the same inputs
    hout = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in dev_out]
    h2d = host_in.numel() * host_in.element_size()
    d2h = dev_out[0].numel() * dev_out[0].element_size()
    sbytes, _ = step_bytes(wl)
    flush_between = sbytes <= L2_BYTES

    def compute(ls):
        if wl.n_append:
            cache.lengths.copy_(base_len)
        if flush_between:
            flush()
        run_step(cache, ls, base_len, wl)

    graphs = []
    for ls in layer_sets:
        compute(ls)
        torch.cuda.synchronize()
        graphs.append(capture(lambda ls=ls: run_step(cache, ls, base_len, wl)))
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in layer_sets]      # inputs of the set are on the device
    done = [torch.cuda.Event() for _ in layer_sets]       # the set's layer calls are done
    drained = [torch.cuda.Event() for _ in layer_sets]    # the set's outputs are on the host

    def run(n, t0=None, t1=None):
        for s in range(n):
            p = s % 2
            with torch.cuda.stream(up):
                if s >= 2:
                    up.wait_event(done[p])                 # step s-2 no longer reads these inputs
                if s == 0 and t0 is not None:
                    t0.record(up)
                dev_in[p].copy_(host_in, non_blocking=True)
                ready[p].record(up)
            stream.wait_event(ready[p])
            if s >= 2:
                stream.wait_event(drained[p])              # step s-2's outputs have left these buffers
            if wl.n_append:
                cache.lengths.copy_(base_len)
            if flush_between:
                flush()
            graphs[p].replay()
            done[p].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(done[p])
                hout[p].copy_(dev_out[p], non_blocking=True)
                drained[p].record(down)
        if t1 is not None:
            down.wait_stream(up)
            t1.record(down)
        torch.cuda.synchronize()

    run(4)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    run(args.steps, t0, t1)
    ms = t0.elapsed_time(t1) / args.steps
    return {"value": wl.B * wl.P / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "l2": ("flushed before each step's layer calls, inside the timed run" if flush_between else
                   "not flushed: a step moves more bytes than the L2 holds"),
            "how": "one pinned host->device copy of every layer's q/iq/w, the layer calls (one CUDA graph per "
                   "buffer set), one device->host copy of every layer's output; two buffer sets alternate "
                   "between steps and the copies run on two copy streams under the neighbouring steps' "
                   "layer calls; whole run from the first input copy to the last output copy, per step"}


# ---------------------------------------------------------------------------
# CPU oracle (the cpu_baseline leg and the --impl reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(wl, seed, max_seconds):
    """Times the oracle on whole query units of sequence 0 (every layer of the
    chain for position 0, scoring split over the host's cores).  Returns
    (units/s, cores, description, seconds)."""
    import numpy as np
    import oracle
    from fp4_compressed_sparse_append_b300 import workloads as W

    cores = os.cpu_count() or 1
    lat, ik = W.cache_rows(wl, seed, 0, device="cpu")
    oc = oracle.Cache(1, wl.capacity, wl.D, wl.DI, key_format=wl.key_format)
    w_ik = W.ikey_projection(wl, seed, device="cpu").numpy() if wl.project else None
    project = oracle.project_ikeys_mx if wl.key_format == "mxfp4" else oracle.project_ikeys

    def keys(rows_bits, given):
        return project(*oracle.quantize_rows(rows_bits), w_ik) if wl.project else given

    oc.append(lat[None].numpy(), keys(lat.numpy(), ik.numpy())[None], threads=cores)
    if wl.n_append:
        app = W.append_rows(wl, seed, device="cpu")
        oc.append(app["rows"][:1].numpy(), keys(app["rows"][0].numpy(), app["ikeys"][0].numpy())[None])
    inputs = [{k: v[:1].numpy() for k, v in W.layer_inputs(wl, seed, li, device="cpu").items()}
              for li in range(len(wl.layers))]
    swa = (W.local_rows(wl, seed, device="cpu")[:1].numpy(), wl.window) if wl.window else None
    done, t0 = 0, time.perf_counter()
    while True:
        oracle.run_chain(oc, wl.layers, inputs, wl.K, wl.scale, P=wl.P, pool_keep=wl.pool_blocks,
                         units=[(0, 0)], score_threads=cores, swa=swa)
        done += 1
        el = time.perf_counter() - t0
        if el > max_seconds or done >= 50:
            break
    sample = ("oracle (plain C, fp64) on %d query unit(s) of sequence 0, position 0, all %d layer(s); "
              "indexer scoring split over %d threads; inputs drawn on the CPU" % (done, len(wl.layers), cores))
    return done / el, cores, sample, el


def bench_reference(args, wl, rank):
    if rank != 0:
        return
    import numpy as np  # noqa: F401
    import oracle
    oracle.build()
    from fp4_compressed_sparse_append_b300 import workloads as W  # noqa: F401
    # warm-up steps, then timed steps; each step = one query unit through the chain
    per_step = []
    cores = os.cpu_count() or 1
    for i in range(args.warmup + args.steps):
        rate, cores, sample, el = oracle_sample(wl, args.seed, 0.0)
        if i >= args.warmup:
            per_step.append(el)
    ms = 1e3 * statistics.mean(per_step)
    value = 1.0 / (ms / 1e3)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(wl),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": "each step: " + sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ---------------------------------------------------------------------------
# Persistent cache records (spill / reload), measured on their own workloads
# ---------------------------------------------------------------------------

PERSIST_METRIC = "cache entries spilled to records and reloaded per second"
PERSIST_WORKLOADS = {
    # one 1M-entry sequence of 512-dim FP4 entries with 128-dim indexer keys
    "persist_1m_mx": dict(B=1, L=1 << 20, D=512, DI=128, key_format="mxfp4"),
    "persist_1m": dict(B=1, L=1 << 20, D=512, DI=128, key_format="e4m3"),
}


def persist_workload(name):
    from fp4_compressed_sparse_append_b300 import workloads as W
    p = PERSIST_WORKLOADS[name]
    return W.Workload(name, B=p["B"], L=p["L"], H=64, D=p["D"], HI=64, DI=p["DI"], K=2048,
                      key_format=p["key_format"])


def persist_config(wl, record_bytes):
    return {"workload": wl.name, "batch": wl.B, "entries_per_sequence": wl.L, "d_latent": wl.D,
            "indexer_dim": wl.DI, "record_bytes": record_bytes,
            "kv_format": "E2M1 codes + E4M3 scale per 16 channels; " + (
                "MXFP4 indexer keys" if wl.key_format == "mxfp4" else "FP8 E4M3 indexer keys"),
            "step": "spill every entry to records, reload them into a second cache",
            "l2": "flushed between timed steps (a 256 MiB read outside the timed events)"}


def persist_oracle_sample(wl, seed, max_seconds, n_sample=1 << 16):
    """The oracle's spill and reload of a window of n_sample entries of sequence 0,
    repeated for about max_seconds.  Returns (entries/s, cores, description, seconds)."""
    import oracle
    from fp4_compressed_sparse_append_b300 import workloads as W
    oracle.build()
    small = wl.scaled(L=n_sample)
    lat, ik = W.cache_rows(small, seed, 0, device="cpu")
    src = oracle.Cache(1, n_sample, wl.D, wl.DI, key_format=wl.key_format)
    src.append(lat[None].numpy(), ik[None].numpy())
    done, t0 = 0, time.perf_counter()
    while True:
        rec = oracle.cache_spill(src, 0, n_sample)
        dst = oracle.Cache(1, n_sample, wl.D, wl.DI, key_format=wl.key_format)
        oracle.cache_reload(dst, rec)
        done += 1
        el = time.perf_counter() - t0
        if el > max_seconds or done >= 1000:
            break
    sample = ("oracle (plain C) spill and reload of %d entries of sequence 0, %d time(s), one thread"
              % (n_sample, done))
    return done * n_sample / el, 1, sample, el


def bench_persist(args, name, rank, world, local_rank):
    import torch
    from fp4_compressed_sparse_append_b300 import binding as B
    from fp4_compressed_sparse_append_b300 import build as BUILD
    from fp4_compressed_sparse_append_b300 import workloads as W

    if rank == 0 or not os.path.exists(BUILD.LIB):
        BUILD.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = persist_workload(name)
    src = B.Cache(wl.B, wl.capacity, wl.D, wl.DI, device=dev, key_format=wl.key_format)
    for b in range(wl.B):
        lat, ik = W.cache_rows(wl, args.seed + rank, b, device=dev)
        one = B.Cache(1, wl.capacity, wl.D, wl.DI, device=dev, key_format=wl.key_format)
        B.csa_quantize_append(one, lat[None], ik[None])
        for t in ("codes", "scales", "ikeys", "iscales"):
            if getattr(one, t) is not None:
                getattr(src, t)[b].copy_(getattr(one, t)[0])
        del one
    src.lengths.fill_(wl.L)
    dst = B.Cache(wl.B, wl.capacity, wl.D, wl.DI, device=dev, key_format=wl.key_format)
    rb = B.csa_cache_record_bytes(src)
    recs = torch.empty((wl.B, wl.L, rb), dtype=torch.uint8, device=dev)
    host = torch.empty((wl.B, wl.L, rb), dtype=torch.uint8).pin_memory()
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    def spill(out):
        B.csa_cache_spill(src, 0, wl.L, records=out)

    def reload(inp):
        dst.lengths.zero_()                     # each step reloads into the same empty cache
        B.csa_cache_reload(dst, inp)

    for _ in range(max(3, args.warmup)):
        spill(recs)
        reload(recs)
    torch.cuda.synchronize()
    for t in ("codes", "scales", "ikeys", "iscales", "lengths"):
        if getattr(src, t) is not None and not torch.equal(getattr(src, t), getattr(dst, t)):
            raise RuntimeError("reloaded cache differs from the spilled one (%s)" % t)
    if B.csa_device_status() != 0:
        raise RuntimeError("device status word set during warm-up")

    def timed_graph(fn, steps):
        g = capture(fn)
        ts = []
        for i in range(steps + 3):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            if i >= 3:
                ts.append((a, b))
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in ts]

    launches0 = B.csa_kernel_launches()
    step_graph = capture(lambda: (spill(recs), reload(recs)))
    launches_per_step = B.csa_kernel_launches() - launches0
    clocks = Clocks(local_rank)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    for i in range(args.steps):
        flush()
        ev[i][0].record(stream)
        step_graph.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    clock_info = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms, value = aggregate_over_ranks(sum(step_ms), wl.B * wl.L, args.steps, world, dev)
    ms_per_step = total_ms / args.steps
    # each kernel alone (the roofline's launch time)
    spill_ms = statistics.mean(timed_graph(lambda: spill(recs), max(3, args.steps)))
    reload_ms = statistics.mean(timed_graph(lambda: reload(recs), max(3, args.steps)))
    # end to end: records in pinned host memory (the spill writes them across
    # the host link, the reload reads them back)
    e2e_ms = statistics.mean(timed_graph(lambda: (spill(host), reload(host)), max(3, args.steps)))
    torch.cuda.synchronize()
    for t in ("codes", "scales", "ikeys", "iscales", "lengths"):
        if getattr(src, t) is not None and not torch.equal(getattr(src, t), getattr(dst, t)):
            raise RuntimeError("reloaded cache differs from the spilled one (%s)" % t)
    if B.csa_device_status() != 0:
        raise RuntimeError("device status word set during the timed region")
    rec_bytes = wl.B * wl.L * rb
    return dict(wl=wl, rb=rb, value=value, ms_per_step=ms_per_step, step_ms=step_ms, clocks=clock_info,
                launches=launches_per_step * args.steps, spill_ms=spill_ms, reload_ms=reload_ms, e2e_ms=e2e_ms,
                rec_bytes=rec_bytes)


def persist_main(args, rank, world, local_rank):
    import json as _json
    r = bench_persist(args, args.workload, rank, world, local_rank)
    if rank != 0:
        return
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = _json.load(f)
    except OSError:
        pass
    peak = peaks.get("hbm_gbs")
    peak_src = "measured (copy bandwidth, burst)" if peak else "fallback"
    peak = peak or 6400.0
    wl, nbytes = r["wl"], r["rec_bytes"]
    # each kernel reads and writes every record's bytes once: 2 x record bytes per entry
    kern = {"spill": r["spill_ms"], "reload": r["reload_ms"]}
    dom = max(kern, key=kern.get)
    achieved = 2 * nbytes / (kern[dom] / 1e3) / 1e9
    roof = {"kernel": dom + "_kernel", "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "peak_source": peak_src, "algorithmic_bytes_per_launch": 2 * nbytes,
            "launch_ms": kern[dom], "traffic": None, "traffic_source": "not captured",
            "other": {k: {"launch_ms": v, "achieved": 2 * nbytes / (v / 1e3) / 1e9} for k, v in kern.items()}}
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        rate, cores, sample, el = persist_oracle_sample(wl, args.seed, 10.0)
        cpu = {"value": rate, "unit": "entries/s", "cores": cores, "kind": "oracle", "sample": sample,
               "seconds": el}
    e2e_value = world * wl.B * wl.L / (r["e2e_ms"] / 1e3)
    line = {
        "metric": PERSIST_METRIC, "value": r["value"], "unit": "entries/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": r["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic (seeded cache rows; no dataset)",
        "config": persist_config(wl, r["rb"]),
        "step_algorithmic_bytes": 4 * nbytes, "hbm_gbs": 4 * nbytes / (r["ms_per_step"] / 1e3) / 1e9,
        "roofline": roof, "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "entries/s", "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes,
                "ms_per_step": r["e2e_ms"], "host_link_gbs": 2 * nbytes / (r["e2e_ms"] / 1e3) / 1e9,
                "how": "spill into pinned host memory and reload from it (the kernels address the host buffer)"},
        "gpu_launches": r["launches"], "clocks": r["clocks"],
    }
    print(json.dumps(line))


def persist_reference(args, rank):
    if rank != 0:
        return
    wl = persist_workload(args.workload)
    per_step, sample, cores = [], "", 1
    for i in range(args.warmup + args.steps):
        rate, cores, sample, el = persist_oracle_sample(wl, args.seed, 0.0)
        if i >= args.warmup:
            per_step.append(el)
    n = 1 << 16
    ms = 1e3 * statistics.mean(per_step)
    value = n / (ms / 1e3)
    from fp4_compressed_sparse_append_b300 import workloads as W  # noqa: F401
    import oracle
    line = {"impl": "reference", "metric": PERSIST_METRIC, "value": value, "unit": "entries/s", "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
            "config": persist_config(wl, oracle.record_bytes(wl.D, wl.DI, wl.key_format)),
            "cpu_baseline": {"value": value, "unit": "entries/s", "cores": cores, "kind": "oracle",
                             "sample": "each step: " + sample},
            "e2e": {"value": value, "unit": "entries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def config_of(wl):
    from fp4_compressed_sparse_append_b300 import workloads as W
    return {"workload": wl.name, "batch": wl.B, "context": wl.L, "query_positions": wl.P, "heads": wl.H,
            "d_latent": wl.D, "indexer_heads": wl.HI, "indexer_dim": wl.DI, "top_k": wl.K,
            "layers": "".join({W.FULL: "F", W.REINDEX: "X", W.REUSE: "R"}[m] for m in wl.layers),
            "pool_blocks": wl.pool_blocks, "appended_rows": wl.n_append,
            "kv_format": "E2M1 codes + E4M3 scale per 16 channels; " + (
                "MXFP4 indexer keys (E2M1 codes + UE8M0 scale per 32 channels)" if wl.key_format == "mxfp4"
                else "FP8 E4M3 indexer keys"),
            "l2": "flushed between timed steps (a 256 MiB read outside the timed events)"}


# Sources whose hash a profile summary records, per stage: the summary's DRAM
# traffic applies only while these files are unchanged.
STAGE_SOURCES = {
    "index_score": ("index_score.cu", "common.cuh"),
    "topk": ("topk.cu", "pool_select.cu", "select_cta.cuh", "common.cuh"),
    "pool_topk": ("pool_select.cu", "select_cta.cuh", "common.cuh"),
    "sparse_attend": ("attend.cu", "common.cuh"),
}


def traffic_from_profile(stage, kind, workload):
    """DRAM bytes per launch of a stage's kernel from the committed ncu summary
    profiles/<stage>_<kind>_<workload>.md, or None where there is none, or when
    the kernel's sources have changed since that capture (the summary records
    the sha256 of the sources it was taken with)."""
    import hashlib
    name = "%s_%s_%s.md" % (stage, kind.replace("+", "_").replace(".", "_"), workload)
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None, "no ncu capture of this stage on this workload"
    csrc = os.path.join(ROOT, "fp4_compressed_sparse_append_b300", "csrc")
    try:
        text = open(path).read()
        h = hashlib.sha256()
        for src in STAGE_SOURCES[stage]:
            with open(os.path.join(csrc, src), "rb") as f:
                h.update(f.read())
    except OSError:
        return None, "no ncu summary"
    want = re.search(r"kernel_sources_sha256:\s*([0-9a-f]{64})", text)
    val = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    if not want or not val:
        return None, "no ncu summary"
    if want.group(1) != h.hexdigest():
        return None, "kernel changed since the ncu capture"
    return int(val.group(1)), "ncu dram__bytes_read.sum + dram__bytes_write.sum (profiles/%s)" % name


def stage_bytes(wl, kind, stage):
    """Algorithmic bytes (bytes that must move) of one launch of a stage:
    index_score: the indexer keys scanned, the indexer queries and weights;
    topk: the scores read (and the pool's block ids) and the ids written; a
    Full layer that builds the pool reads its blocks' maxima (L/8) and the
    pool's rows' scores instead of all L scores;
    pool_topk (index_score and topk of a Reindex layer in one kernel): the
    pool's block ids and keys, the indexer queries and weights, the ids;
    sparse_attend: the selected FP4 rows, the bf16 queries, the fp32 outputs
    and log-sum-exps (and the local window's FP8 rows)."""
    from fp4_compressed_sparse_append_b300 import workloads as W
    units = wl.B * wl.P
    L = wl.length_after_append
    kb = W.key_bytes(wl)
    pool_rows = wl.pool_blocks * 8
    q_index = units * wl.HI * (wl.DI + 4)
    if stage == "index_score":
        keys = units * pool_rows * kb if kind == "reindex.pool" else wl.B * L * kb
        return keys + q_index
    if stage == "pool_topk":
        # the pool's block ids and its rows' keys read, the ids written
        return units * (wl.pool_blocks * 4 + pool_rows * kb + wl.K * 4) + q_index
    if stage == "topk":
        if kind == "full+pool":
            # the block maxima, the pool's rows' scores, the pool written, the ids
            return units * (((L + 7) // 8) * 4 + pool_rows * 4 + wl.pool_blocks * 4 + wl.K * 4)
        n = pool_rows if kind == "reindex.pool" else L
        b = units * n * 4 + units * wl.K * 4
        if kind == "reindex.pool":
            b += units * wl.pool_blocks * 4
        return b
    row = wl.D // 2 + wl.D // 16
    b = units * (min(wl.K, L) * row + wl.H * wl.D * (2 + 4) + wl.H * 4)
    if wl.window:
        b += wl.B * (wl.window + wl.P - 1) * wl.D
    return b


KERNELS = {"index_score": "index_score_kernel", "topk": "select_kernel (+ select_one_kernel, pool_rows_kernel)",
           "pool_topk": "pool_spread_kernel", "sparse_attend": "attend_kernel (+ attend_merge_kernel)"}


def stage_rooflines(wl, stages, peak_hbm, peak_src, peak_tf, peak_tf_src):
    """Roofline of every timed stage against HBM (the bound of every workload
    but the multi-position verify ones, whose attention is reported against the
    tensor cores: S = Q.V^T and O = P.V, 2*H*D flops each per selected row and
    query, fp16 operands at the dense bf16 rate)."""
    out = {}
    for name, st in stages.items():
        ms = st["ms"]
        stage = st["stage"]
        nbytes = stage_bytes(wl, st["kind"], stage)
        traffic, traffic_src = traffic_from_profile(stage, st["kind"], wl.name)
        r = {"kernel": KERNELS[stage], "launches_per_step": st["launches"], "launch_ms": ms,
             "share_of_stage_time": None, "algorithmic_bytes_per_launch": nbytes,
             "traffic": traffic, "traffic_source": traffic_src}
        if stage == "sparse_attend" and wl.P > 1:
            flops = wl.B * wl.P * 4.0 * wl.H * min(wl.K, wl.length_after_append) * wl.D
            ach = flops / (ms / 1e3) / 1e12
            r.update(bound="tensor", achieved=ach, peak=peak_tf, unit="TFLOP/s", frac=ach / peak_tf,
                     peak_source=peak_tf_src + " (bf16 dense, burst)", algorithmic_flops_per_launch=flops)
        else:
            ach = nbytes / (ms / 1e3) / 1e9
            r.update(bound="hbm", achieved=ach, peak=peak_hbm, unit="GB/s", frac=ach / peak_hbm,
                     peak_source=peak_src + " (copy bandwidth, burst)")
        out[name] = r
    total = sum(st["ms"] * st["launches"] for st in stages.values())
    for name, st in stages.items():
        out[name]["share_of_stage_time"] = st["ms"] * st["launches"] / total if total else None
    return out


def main():
    args = parse_args()
    rank, world, local_rank = dist_env()
    from fp4_compressed_sparse_append_b300 import workloads as W
    if args.workload in PERSIST_WORKLOADS:
        if args.impl == "reference":
            persist_reference(args, rank)
            return
        if world > 1:
            import torch
            import torch.distributed as dist
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
        persist_main(args, rank, world, local_rank)
        return
    wl = W.WORKLOADS[args.workload]
    if args.impl == "reference":
        bench_reference(args, wl, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    r = bench_ours(args, wl, rank, world, local_rank)
    if rank != 0:
        return
    import json as _json
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = _json.load(f)
    except OSError:
        pass
    peak_hbm = peaks.get("hbm_gbs")
    peak_src = "measured" if peak_hbm else "fallback"
    peak_hbm = peak_hbm or 6400.0
    peak_tf = peaks.get("bf16_tflops")
    peak_tf_src = "measured" if peak_tf else "fallback"
    peak_tf = peak_tf or 1800.0
    # The dominant kernel: the stage with the largest time per step (its time
    # alone times its launches per step).
    stages = r["stages"]
    dominant = max(stages, key=lambda k: stages[k]["ms"] * stages[k]["launches"]) if stages else None
    rooflines = stage_rooflines(wl, stages, peak_hbm, peak_src, peak_tf, peak_tf_src)
    roof = rooflines.get(dominant)
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        rate, cores, sample, el = oracle_sample(wl, args.seed, 20.0)
        cpu = {"value": rate * wl.P, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample,
               "seconds": el}
    line = {
        "metric": METRIC, "value": r["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": r["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3/e2m1 operands, f32 accumulate",
        "data": "synthetic (seeded draws shaped like the workload; no dataset)",
        "config": config_of(wl),
        "hbm_gbs": r["gbs"], "frac_of_8tbs": r["gbs"] / NOMINAL_HBM_GBS, "frac_of_measured_hbm": r["gbs"] / peak_hbm,
        "step_algorithmic_bytes": r["step_bytes"],
        "stages_ms": {k: v["ms"] for k, v in stages.items()}, "dominant_stage": dominant,
        "layers_ms": {"modes": [W.MODE_NAMES[m] for m in wl.layers], "ms": r["layer_ms"],
                      "how": "each layer alone as a graph, L2 flushed before each replay"},
        "roofline": roof, "roofline_stages": rooflines, "cpu_baseline": cpu, "e2e": r["e2e"], "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
