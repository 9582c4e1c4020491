#!/usr/bin/env python3
"""Benchmark of the CSA2 global-attention layer on one GB300.

Default workload (the headline metric): decode at 1,048,576 cached entries per
sequence, batch 16, one 4-layer decoder block = a Reindex layer (own index
queries score only the 2048-block candidate pool, top-512) followed by three
Reuse layers (attention only, same selection and cache, fresh queries).  The
pool comes from a Full source-layer scan done before timing.

Cold-L2 layers: real models run MoE between layers, so a layer's cache reads
come from HBM.  The bench keeps R independent batches (instances, each with its
own 5.97 GB cache copy) and software-pipelines them: step s runs the Reindex
layer of instance s, Reuse-1 of instance s-d, Reuse-2 of s-2d and Reuse-3 of
s-3d, so roughly d steps (d * 44 MB > L2) pass between two layers touching
the same instance.  One step = four layer calls of batch 16 = 64
query-token-layers.  The four calls of a step belong to four different
instances, so they are independent and run as parallel branches of the step's
CUDA graph (four streams); the line also reports the same steps with the calls
in sequence on one stream (``serial_schedule``).

``--seq-len`` shrinks the cache (the same step on fewer entries; used for
small profiler captures), ``--cpu-sample-queries 0`` skips the CPU oracle leg.

``--impl reference`` times the CPU oracle (the checker, not a product path) on
a bounded sample of the same workload.

The roofline's ``traffic`` (DRAM bytes per launch of the dominant kernel) is
read from the ncu summary under ``profiles/`` and reported only while the
kernel's source file still has the hash recorded beside the figure.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CSA2 decode query-tokens/s/layer at 1M ctx; % of HBM roofline"
UNIT = "query-token-layers/s"

# algorithmic bytes (per query token) of the 1M Reindex + 3 Reuse chain: what the
# layer must read and write (pool entries, ids, queries, weights, selection,
# the selected entries, the window, q and out), nothing of this implementation's own
IDX_ENTRY, MAIN_ENTRY = 68, 288
K_SEL, M_BLK, WIN, D, H, HI, DI = 512, 2048, 128, 512, 64, 32, 128
ATTN_BYTES = K_SEL * MAIN_ENTRY + WIN * D * 2 + H * D * 2 + H * D * 2          # 409,600
REINDEX_BYTES = M_BLK * 8 * IDX_ENTRY + M_BLK * 4 + HI * DI * 2 + HI * 4 + K_SEL * 4 + ATTN_BYTES   # 1,542,272
REUSE_BYTES = K_SEL * 4 + ATTN_BYTES                                             # 411,648
CHAIN_BYTES = REINDEX_BYTES + 3 * REUSE_BYTES                                    # 2,777,216
# traffic this implementation adds: the Reindex call writes a packed copy of its
# selected entries (K x 288 B per query), which the Reuse calls read in place of
# the gather (so their byte count is unchanged)
PACKED_WRITE_BYTES = K_SEL * MAIN_ENTRY                                          # 147,456

# the K-step window is replayed back to back until at least this long, and the
# median window is reported (steady state, not a single fill and drain)
MIN_TIMED_S = 0.5


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def ncu_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from profiles/traffic.txt, or None when
    absent or when the kernel's source changed since the capture."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.txt")) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 4 and parts[0] == kernel and not line.startswith("#"):
                    src = os.path.join(ROOT, "fp4_kv_cache_csa2_gb300", "csrc", parts[2])
                    with open(src, "rb") as g:
                        if hashlib.sha256(g.read()).hexdigest()[:16] == parts[3]:
                            return float(parts[1])
    except OSError:
        pass
    return None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append([x.strip() for x in line.split(",")])

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(s[0]) for s in self.samples if s[0].replace('.', '').isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace('.', '').isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for s in self.samples:
            for name, v in zip(names, s[3:7]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(self.samples)}


# ------------------------------------------------------------------ helpers
def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest value over the ranks (the job's time is its slowest replica's)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ decode 1M
class Decode1M:
    """Reindex + 3 Reuse at 1,048,576 entries, batch 16, R pipelined instances."""

    def __init__(self, csa2, torch, B=16, N=1 << 20, d=3, seed=3, lanes=2, packed=True, swa_fp8=False):
        import synth
        self.csa2, self.torch = csa2, torch
        self.swa_fp8 = swa_fp8
        self.B, self.N, self.d = B, N, d
        self.R = 3 * d + 1
        dev = "cuda"
        self.stream = torch.cuda.current_stream()
        t0 = time.time()
        # ---- instance 0's cache from seeded N(0,1) latents through the cache write (m = 1)
        base = csa2.Cache(B, N, 1, device=dev)
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        w_idx = synth.torch_normal(seed + 1, (DI, D), torch.float32, dev).mul_(1 / math.sqrt(D)).to(torch.bfloat16)
        rope = csa2.rope_table(N).to(dev)
        ws_cw = csa2.Workspace(1 << 16, device=dev)
        chunk = min(1 << 17, N)
        ones = torch.ones(D, device=dev)
        for b in range(B):
            for c0 in range(0, N, chunk):
                x = torch.randn((1, chunk, D), generator=g, device=dev).to(torch.bfloat16)
                start = torch.tensor([c0], dtype=torch.int64, device=dev)
                cache_b = base.sequence(b)
                csa2.compress_quantize(cache_b, x.view(torch.int16), start, ones, ones, rope, w_idx.view(torch.int16),
                                       ws_cw)
        base.n_entries.fill_(N)
        del rope
        torch.cuda.synchronize()
        assert ws_cw.sync_status()[0] == 0
        self.setup_cache_s = time.time() - t0
        # ---- candidate pool: one untimed Full source-layer scan of instance 0 (own index queries)
        M, K = M_BLK, K_SEL
        self.q_pos = torch.full((B, 1), N - 1, dtype=torch.int64, device=dev)
        self.swa_base = torch.full((B,), N - WIN, dtype=torch.int64, device=dev)
        full_q_idx = synth.torch_normal(seed + 2, (B, 1, HI, DI), torch.bfloat16, dev)
        full_w = synth.torch_normal(seed + 3, (B, 1, HI), torch.float32, dev)
        full_q = synth.torch_normal(seed + 4, (B, 1, H, D), torch.bfloat16, dev)
        full_swa = synth.torch_swa_rows(seed + 5, (B, WIN), dev)
        self.pool = torch.empty((B, 1, M), dtype=torch.int32, device=dev)
        sel0 = torch.empty((B, 1, K), dtype=torch.int32, device=dev)
        out0 = torch.empty((B, 1, H, D), dtype=torch.bfloat16, device=dev)
        ws_full = csa2.Workspace(csa2.decode_workspace_size(csa2.MODE_FULL, B, 1, N, M, K), device=dev)
        t1 = time.time()
        csa2.decode(csa2.MODE_FULL, base, q_pos=self.q_pos, q=full_q.view(torch.int16), swa=full_swa.view(torch.int16),
                    swa_base_pos=self.swa_base, scale=1 / math.sqrt(D), sel=sel0, out=out0.view(torch.int16),
                    ws=ws_full, M=M, max_n=N, q_idx=full_q_idx.view(torch.int16), w_head=full_w,
                    pool_blocks=self.pool)
        torch.cuda.synchronize()
        self.full_scan_ms = (time.time() - t1) * 1e3
        assert ws_full.sync_status()[0] == 0
        del ws_full
        # ---- R instances: cache copies at distinct addresses, own queries per layer
        self.caches = [base] + [_clone_cache(base) for _ in range(self.R - 1)]
        self.inst = []
        for r in range(self.R):
            s = seed + 100 * (r + 1)
            inst = {
                "q_idx": synth.torch_normal(s + 1, (B, 1, HI, DI), torch.bfloat16, dev),
                "w_head": synth.torch_normal(s + 2, (B, 1, HI), torch.float32, dev),
                "q": [synth.torch_normal(s + 10 + l, (B, 1, H, D), torch.bfloat16, dev) for l in range(4)],
                "swa": [synth.torch_swa_rows(s + 20 + l, (B, WIN), dev) for l in range(4)],
                "out": [torch.empty((B, 1, H, D), dtype=torch.bfloat16, device=dev) for l in range(4)],
                "sel": torch.empty((B, 1, K), dtype=torch.int32, device=dev),
                # the selected entries packed by the Reindex call, read by the Reuse calls
                "packed": torch.empty((B, 1, K, MAIN_ENTRY), dtype=torch.uint8, device=dev) if packed else None,
            }
            if swa_fp8:          # the window rows stored as E4M3, quantised once
                inst["swa8"] = [torch.empty((B, WIN, D), dtype=torch.uint8, device=dev) for _ in range(4)]
                for l in range(4):
                    csa2.swa_quantize_fp8(inst["swa"][l].view(torch.int16), inst["swa8"][l])
            self.inst.append(inst)
        # one workspace per layer slot: the four layer calls of a step may run at once
        # lanes per layer slot (stream + workspace), taken by step number modulo the
        # lane count, so that the same layer's calls of consecutive steps (different
        # instances) can overlap
        self.lanes = lanes
        self.ws = [[csa2.Workspace(csa2.decode_workspace_size(csa2.MODE_REINDEX if l == 0 else csa2.MODE_REUSE,
                                                              B, 1, N, M, K), device=dev) for _ in range(self.lanes)]
                   for l in range(4)]
        # the Reindex branch (fused score/select + attention) is the step's critical
        # path: it runs on a high-priority stream and is enqueued first
        self.hi = [torch.cuda.Stream(priority=-1) for _ in range(self.lanes)]
        self.side = [[torch.cuda.Stream() for _ in range(self.lanes)] for _ in range(3)]
        for r in range(self.R):          # every instance starts with a published selection
            self.layer(0, r)
        torch.cuda.synchronize()
        self.check_status()
        self.setup_s = time.time() - t0

    def stream_of(self, layer: int, s: int):
        return (self.hi if layer == 0 else self.side[layer - 1])[s % self.lanes]

    def all_streams(self):
        return [*self.hi, *(st for lane in self.side for st in lane)]

    def layer(self, layer: int, r: int, lane: int = 0):
        csa2, inst, torch = self.csa2, self.inst[r], self.torch
        mode = csa2.MODE_REINDEX if layer == 0 else csa2.MODE_REUSE
        swa = inst["swa8"][layer] if self.swa_fp8 else inst["swa"][layer].view(torch.int16)
        csa2.decode(mode, self.caches[r], q_pos=self.q_pos, q=inst["q"][layer].view(torch.int16),
                    swa=swa, swa_base_pos=self.swa_base, scale=1 / math.sqrt(D),
                    sel=inst["sel"], out=inst["out"][layer].view(torch.int16), ws=self.ws[layer][lane], M=M_BLK,
                    max_n=self.N, packed_sel=inst["packed"], swa_fp8=self.swa_fp8,
                    q_idx=inst["q_idx"].view(torch.int16), w_head=inst["w_head"], pool_blocks=self.pool)

    def check_status(self):
        for ws in (w for lane in self.ws for w in lane):
            st, detail = ws.sync_status()
            assert st == 0, f"device status {st} ({detail})"

    def step(self, s: int, concurrent: bool = True):
        """Reindex(s), Reuse1(s-d), Reuse2(s-2d), Reuse3(s-3d) over instances mod R.
        The four calls touch four different instances (R > 3d), so they are
        independent: concurrently they run as parallel branches (the Reindex call
        on the current stream, the Reuse calls on three side streams), otherwise
        one after another on the current stream."""
        torch = self.torch
        if not concurrent:
            for layer in range(4):
                self.layer(layer, (s - layer * self.d) % self.R)
            return
        main = torch.cuda.current_stream()
        fork = torch.cuda.Event()
        fork.record(main)
        lane = s % self.lanes
        for layer in range(4):
            st = self.stream_of(layer, s)
            st.wait_event(fork)
            with torch.cuda.stream(st):
                self.layer(layer, (s - layer * self.d) % self.R, lane)
        for layer in range(4):
            join = torch.cuda.Event()
            join.record(self.stream_of(layer, s))
            main.wait_event(join)

    def cycle(self, s_base: int, n_steps: int = 0):
        """Steps s_base .. s_base + n_steps - 1 (default R) with only the dependencies the data
        imposes, so that consecutive steps overlap: every layer slot keeps its
        own stream (and workspace) across the steps, a Reuse-k call waits for
        the Reindex call that produced its instance's selection (step s - 3k
        wrote it), and a Reindex call waits for the three Reuse calls that read
        its instance's previous selection (steps s - R + 3k)."""
        torch = self.torch
        main = torch.cuda.current_stream()
        streams = self.all_streams()
        fork = torch.cuda.Event()
        fork.record(main)
        for st in streams:
            st.wait_event(fork)
        done = {}
        for i in range(n_steps or self.R):
            s = s_base + i
            for layer in range(4):
                st = self.stream_of(layer, s)
                if layer > 0:
                    dep = [(0, s - layer * self.d)]
                else:
                    dep = [(k, s - self.R + k * self.d) for k in range(1, 4)]
                for key in dep:
                    if key in done:
                        st.wait_event(done[key])
                with torch.cuda.stream(st):
                    self.layer(layer, (s - layer * self.d) % self.R, s % self.lanes)
                ev = torch.cuda.Event()
                ev.record(st)
                done[(layer, s)] = ev
        for st in streams:
            join = torch.cuda.Event()
            join.record(st)
            main.wait_event(join)

    def prologue(self):
        for s in range(3 * self.d):
            self.step(s)


def latency_split(torch, B: int, Q: int, K: int = K_SEL) -> int:
    """CTAs per query in the attention of a call that runs alone (one call at a
    time, so one CTA per query would leave most SMs idle): as many as keep the
    call within one wave, at most one per key chunk (the window and every run
    of 128 selected entries), and none (1) unless that is at least 3 (64
    queries split in 2 were slower than one CTA each) or above the library's
    split limit."""
    bq = B * Q
    if bq > 128:
        return 1
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    s = min(1 + -(-K // 128), sms // bq)
    return s if s >= 3 else 1


def _clone_cache(c):
    import fp4_kv_cache_csa2_gb300 as csa2
    n = csa2.Cache.__new__(csa2.Cache)
    n.B, n.cap, n.m = c.B, c.cap, c.m
    n.main_kv = c.main_kv.clone()
    n.idx_codes = c.idx_codes.clone()
    n.idx_scales = c.idx_scales.clone()
    n.n_entries = c.n_entries.clone()
    return n


def _capture(torch, fn):
    """CUDA graph of the launches `fn` enqueues (the library calls only enqueue)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


class PhaseGraphs:
    """CUDA graphs of a pipelined step: one per pipeline phase (step s depends
    only on s mod R), one of a whole cycle of R consecutive steps starting at
    each phase, and optionally one of `cycles` whole cycles starting at each
    phase, so that a run of steps launches one graph per cycle (or per
    `cycles` cycles) whatever phase it starts at (consecutive graph launches
    serialise, so every graph boundary is a drain and fill of the pipeline)."""

    def __init__(self, torch, step_fn, R: int, s_base: int, cycle_fn=None, cycles: int = 1):
        self.R = R
        self.cycles = max(1, cycles)
        self.single = [_capture(torch, lambda i=i: step_fn(s_base + i)) for i in range(R)]
        if cycle_fn is None:
            cycle_fn = lambda first, n: [step_fn(first + i) for i in range(n)]
        self.cycle_at = [_capture(torch, lambda p=p: cycle_fn(s_base + p, R)) for p in range(R)]
        self.multi_at = ([_capture(torch, lambda p=p: cycle_fn(s_base + p, R * self.cycles)) for p in range(R)]
                         if self.cycles > 1 else None)

    def run(self, first: int, n: int):
        """Replays steps first .. first + n - 1 (exactly n steps)."""
        i = 0
        long = self.R * self.cycles
        while i < n:
            p = (first + i) % self.R
            if self.multi_at is not None and n - i >= long:
                self.multi_at[p].replay()
                i += long
            elif n - i >= self.R:
                self.cycle_at[p].replay()
                i += self.R
            else:
                self.single[p].replay()
                i += 1


def steady_windows(torch, run_window, n_steps, first, min_s=MIN_TIMED_S, max_windows=20000):
    """Times the same K-step window (run_window(first_step, K) enqueues exactly K
    steps) replayed back to back: a CUDA event before the first window and after
    each one, all on the current stream, one synchronize at the end.  The number
    of windows is chosen from one calibration window so the whole set lasts at
    least `min_s`.  Returns (median ms per window, windows, total seconds)."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    run_window(first, n_steps)
    e1.record()
    torch.cuda.synchronize()
    cal = max(e0.elapsed_time(e1), 1e-3)
    n_win = int(min(max_windows, max(5, math.ceil(min_s * 1e3 / cal))))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_win + 1)]
    s = first + n_steps
    torch.cuda.synchronize()
    ev[0].record()
    for w in range(n_win):
        run_window(s + w * n_steps, n_steps)
        ev[w + 1].record()
    torch.cuda.synchronize()
    times = [ev[w].elapsed_time(ev[w + 1]) for w in range(n_win)]
    return statistics.median(times), n_win, ev[0].elapsed_time(ev[-1]) / 1e3


def _graph_ms(torch, graph, reps):
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    graph.replay()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(reps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def graph_cycles(args, R: int) -> int:
    """Pipeline cycles per replayed graph: --graph-cycles, or (0) as many whole
    cycles as a timed window of --steps steps holds, at most 10, so that a
    window replays as few graphs as possible (each graph boundary drains the
    pipeline: at --steps 20, graphs of 20 steps measured 2.18M against 2.03M
    with graphs of 10)."""
    if args.graph_cycles > 0:
        return args.graph_cycles
    return max(1, min(10, args.steps // R))


def run_decode1m(args, torch, csa2):
    rank, world, local = dist_info()
    fp8 = args.swa_format == "fp8"
    w = Decode1M(csa2, torch, N=args.seq_len, d=args.pipeline_distance, lanes=args.lanes,
                 packed=bool(args.packed_selection), swa_fp8=fp8)
    w.prologue()
    torch.cuda.synchronize()
    # graphs per pipeline phase and per cycle of R phases: step s only depends on s mod R
    s_base = 3 * w.d
    cycles = graph_cycles(args, w.R)
    graphs = PhaseGraphs(torch, w.step, w.R, s_base, cycle_fn=w.cycle, cycles=cycles)
    n_steps = args.steps
    s0 = args.warmup
    with ClockSampler(local) as clk:             # sampling from the warm-up on
        graphs.run(0, args.warmup)
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("timed")
        win_ms, n_win, timed_s = steady_windows(torch, graphs.run, n_steps, s0)
        torch.cuda.nvtx.range_pop()
        barrier(world)
    total_ms = max_over_ranks(win_ms, world)
    w.check_status()
    # the same steps with the four layer calls one after another on one stream
    serial = PhaseGraphs(torch, lambda s: w.step(s, concurrent=False), w.R, s_base)
    serial.run(0, args.warmup)
    torch.cuda.synchronize()
    n_serial = min(n_steps, 1000)
    serial_win, _, _ = steady_windows(torch, serial.run, n_serial, s0, min_s=0.2)
    serial_ms = max_over_ranks(serial_win, world) / n_serial
    w.check_status()
    # per-layer-call durations, same pipeline (cold instances), timed by layer type
    reindex_g = _capture(torch, lambda: [w.layer(0, r) for r in range(w.R)])
    reuse_g = _capture(torch, lambda: [w.layer(1 + (r % 3), r) for r in range(w.R)])
    reindex_ms = _graph_ms(torch, reindex_g, 20) / w.R
    reuse_ms = _graph_ms(torch, reuse_g, 20) / w.R
    w.check_status()

    ms_step = total_ms / n_steps
    qtl_per_step = w.B * 4
    value = qtl_per_step * world / (ms_step / 1e3)
    hbm, bf16, which = peaks()
    win_saved = WIN * D if fp8 else 0                  # an E4M3 window row is 512 B, a bf16 one 1 KB
    bytes_step = w.B * (CHAIN_BYTES - 4 * win_saved)
    extra_step = w.B * PACKED_WRITE_BYTES if args.packed_selection else 0
    dom_is_reuse = 3 * reuse_ms >= reindex_ms          # Reuse calls are 3 of the 4 layers
    dom_ms = reuse_ms if dom_is_reuse else reindex_ms
    dom_bytes = w.B * ((REUSE_BYTES if dom_is_reuse else REINDEX_BYTES) - win_saved)
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    dom_kernel = "attn_stream_kernel" if dom_is_reuse else "reindex_select_kernel"
    traffic = ncu_traffic(dom_kernel + (":fp8_window" if fp8 else "")) if w.N == 1 << 20 else None
    e2e = None if fp8 else run_decode1m_e2e(args, torch, csa2, w)
    return {
        "value": value, "ms_per_step": ms_step, "dtype": "fp4-e2m1 cache, mxfp4 index, f16 mma fp32 acc",
        "config": {"workload": f"decode Reindex + 3 Reuse, {w.N:,} entries/seq, batch 16 per layer call",
                   "global_batch": w.B, "seq_len": w.N, "M_blocks": M_BLK, "K": K_SEL, "window": WIN,
                   "window_rows": "E4M3, 512 B per row" if fp8 else "bf16, 1 KB per row",
                   "l2": f"inputs larger than L2: {w.R} pipelined instances x "
                         f"{w.B * w.N * (MAIN_ENTRY + IDX_ENTRY) / 1e9:.2f} GB, layer distance {w.d} steps",
                   "launch": f"CUDA graphs of {w.R * cycles} consecutive steps "
                             f"({cycles} whole cycles of {w.R} from any phase; one graph per step for a remainder) "
                             "with only the data's "
                             "dependencies between steps; in a step the 4 layer calls (4 different pipelined "
                             "instances, so independent) are parallel branches, the Reindex branch first at high "
                             f"priority; every layer slot has {w.lanes} stream + workspace lanes taken by step "
                             f"number mod {w.lanes}",
                   "selection": ("the Reindex call writes a packed copy of its selected entries (K x 288 B per "
                                 "query), which the three Reuse calls read contiguously instead of gathering"
                                 if args.packed_selection else "every layer gathers the selected entries"),
                   "parallelism": "replicas" if world > 1 else "single-gpu"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": traffic,
                     "kernel": dom_kernel + (" (Reuse layer)" if dom_is_reuse else " (Reindex layer)"),
                     "algorithmic_bytes_per_launch": dom_bytes, "avg_launch_ms": dom_ms,
                     "peak_source": which},
        "step_hbm": {"algorithmic_bytes": bytes_step, "GB_s": bytes_step / (ms_step / 1e3) / 1e9,
                     "frac": bytes_step / (ms_step / 1e3) / 1e9 / hbm,
                     "packed_selection_write_bytes": extra_step,
                     "note": "algorithmic bytes of the chain (pool, ids, queries, weights, selection, selected "
                             "entries, window, q, out); the packed-selection write is this implementation's "
                             "own extra traffic, shown apart and not counted"},
        "timing": {"windows": n_win, "steps_per_window": n_steps, "timed_s": timed_s,
                   "how": "the K-step window replayed back to back (CUDA events between windows on the "
                          "launching stream, one synchronize after the set, barrier on both sides); the "
                          "median window / K is ms_per_step"},
        "layer_ms": {"reindex": reindex_ms, "reuse": reuse_ms},
        "serial_schedule": {"value": qtl_per_step * world / (serial_ms / 1e3), "ms_per_step": serial_ms,
                            "steps": n_serial, "launch": "the same graphs with the 4 layer calls in sequence "
                                                         "on one stream"},
        "full_scan_1m_ms_untimed_setup": w.full_scan_ms,
        "clocks": clk.summary(),
        # Reindex layer: fused score + select kernel and attention; Reuse: attention
        "gpu_launches": n_steps * (2 + 3),
        "e2e": e2e,
    }


def run_decode1m_e2e(args, torch, csa2, w):
    """Same pipeline through the public API with the host in the loop.  A step's
    inputs (the four layers' queries, one new window row per sequence and layer,
    the Reindex layer's index queries and head weights) travel in one pinned
    host block and one copy; the four layers' outputs come back in one copy into
    one pinned block.  Serving-style overlap: while step s computes from staging
    buffer s % NB, a copy stream brings step s+1's inputs into the next buffer
    and a second copy stream returns step s-1's outputs, so every timed step
    carries one full input copy and one full output copy.  NB (the lane count,
    else 2) divides R, so a graph of whole phases uses the same buffers on every
    replay."""
    B = w.B
    NB = w.lanes if w.lanes >= 2 and w.R % w.lanes == 0 else 2
    assert w.R % NB == 0
    q_bytes = B * H * D * 2
    row_bytes = B * D * 2
    qidx_bytes = B * HI * DI * 2
    wh_bytes = B * HI * 4
    off_q, off_row = 0, 4 * q_bytes
    off_qidx = off_row + 4 * row_bytes
    off_w = off_qidx + qidx_bytes
    in_bytes = off_w + wh_bytes
    out_bytes = 4 * q_bytes
    host_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    host_out = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
    host_in.view(torch.int16).random_(-16000, 16000)       # bf16 bit patterns of moderate magnitude
    host_in[off_w:].view(torch.float32).normal_()
    dev_in = [torch.empty(in_bytes, dtype=torch.uint8, device="cuda") for _ in range(NB)]
    dev_out = [torch.zeros(out_bytes, dtype=torch.uint8, device="cuda") for _ in range(NB)]
    for t in dev_in:
        t.copy_(host_in)

    def views(k):
        d = dev_in[k]
        return ([d[off_q + l * q_bytes: off_q + (l + 1) * q_bytes].view(torch.int16).view(B, 1, H, D) for l in range(4)],
                [d[off_row + l * row_bytes: off_row + (l + 1) * row_bytes].view(torch.int16).view(B, D)
                 for l in range(4)],
                d[off_qidx: off_qidx + qidx_bytes].view(torch.int16).view(B, 1, HI, DI),
                d[off_w: off_w + wh_bytes].view(torch.float32).view(B, 1, HI),
                [dev_out[k][l * q_bytes:(l + 1) * q_bytes].view(torch.int16).view(B, 1, H, D) for l in range(4)])
    bufs = [views(k) for k in range(NB)]
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()

    def step(s):
        main = torch.cuda.current_stream()          # the capturing stream when captured
        k = s % NB
        q_view, row_view, qidx_view, w_view, out_view = bufs[k]
        fork = torch.cuda.Event()
        fork.record(main)
        h2d.wait_event(fork)
        d2h.wait_event(fork)
        with torch.cuda.stream(h2d):
            dev_in[(s + 1) % NB].copy_(host_in, non_blocking=True)   # inputs of step s + 1
        with torch.cuda.stream(d2h):
            host_out.copy_(dev_out[(s - 1) % NB], non_blocking=True) # outputs of step s - 1
        def layer_call(layer):
            r = (s - layer * w.d) % w.R
            inst = w.inst[r]
            inst["swa"][layer][:, WIN - 1].view(torch.int16).copy_(row_view[layer])
            mode = csa2.MODE_REINDEX if layer == 0 else csa2.MODE_REUSE
            csa2.decode(mode, w.caches[r], q_pos=w.q_pos, q=q_view[layer], swa=inst["swa"][layer].view(torch.int16),
                        swa_base_pos=w.swa_base, scale=1 / math.sqrt(D), sel=inst["sel"], out=out_view[layer],
                        ws=w.ws[layer][s % w.lanes], M=M_BLK, max_n=w.N, q_idx=qidx_view, w_head=w_view,
                        pool_blocks=w.pool, packed_sel=inst["packed"])
        for layer in range(4):                     # independent instances: parallel branches,
            st = w.stream_of(layer, s)             # the Reindex branch first and at high priority
            st.wait_event(fork)
            with torch.cuda.stream(st):
                layer_call(layer)
        for st in (h2d, d2h, *(w.stream_of(layer, s) for layer in range(4))):
            join = torch.cuda.Event()
            join.record(st)
            main.wait_event(join)

    def cycle(s_base, n_steps=0):
        """Steps s_base .. s_base + n_steps - 1 (default R) with only the data's dependencies (see Decode1M.cycle), plus
        the staging buffers': the layer calls of step s wait for the copy that
        brought their inputs (issued during step s - 1) and for the copy-out of
        step s - NB (which read the output block they overwrite); the input copy
        issued during step s waits for step s + 1 - NB's calls (which read that
        buffer) and the output copy for step s - 1's calls."""
        main = torch.cuda.current_stream()
        streams = w.all_streams()
        fork = torch.cuda.Event()
        fork.record(main)
        for st in (*streams, h2d, d2h):
            st.wait_event(fork)
        done, h2d_done, d2h_done = {}, {}, {}
        for i in range(n_steps or w.R):
            s = s_base + i
            k = s % NB
            q_view, row_view, qidx_view, w_view, out_view = bufs[k]
            for l in range(4):
                if (l, s + 1 - NB) in done:
                    h2d.wait_event(done[(l, s + 1 - NB)])
                if (l, s - 1) in done:
                    d2h.wait_event(done[(l, s - 1)])
            with torch.cuda.stream(h2d):
                dev_in[(s + 1) % NB].copy_(host_in, non_blocking=True)   # inputs of step s + 1
            e = torch.cuda.Event()
            e.record(h2d)
            h2d_done[s + 1] = e
            with torch.cuda.stream(d2h):
                host_out.copy_(dev_out[(s - 1) % NB], non_blocking=True) # outputs of step s - 1
            e = torch.cuda.Event()
            e.record(d2h)
            d2h_done[s - 1] = e
            for layer in range(4):
                st = w.stream_of(layer, s)
                dep = [(0, s - layer * w.d)] if layer > 0 else [(kk, s - w.R + kk * w.d) for kk in range(1, 4)]
                for key in dep:
                    if key in done:
                        st.wait_event(done[key])
                if s in h2d_done:
                    st.wait_event(h2d_done[s])
                if s - NB in d2h_done:
                    st.wait_event(d2h_done[s - NB])
                r = (s - layer * w.d) % w.R
                inst = w.inst[r]
                with torch.cuda.stream(st):
                    inst["swa"][layer][:, WIN - 1].view(torch.int16).copy_(row_view[layer])
                    mode = csa2.MODE_REINDEX if layer == 0 else csa2.MODE_REUSE
                    csa2.decode(mode, w.caches[r], q_pos=w.q_pos, q=q_view[layer],
                                swa=inst["swa"][layer].view(torch.int16), swa_base_pos=w.swa_base,
                                scale=1 / math.sqrt(D), sel=inst["sel"], out=out_view[layer],
                                ws=w.ws[layer][s % w.lanes],
                                M=M_BLK, max_n=w.N, q_idx=qidx_view, w_head=w_view, pool_blocks=w.pool,
                                packed_sel=inst["packed"])
                ev = torch.cuda.Event()
                ev.record(st)
                done[(layer, s)] = ev
        for st in (*streams, h2d, d2h):
            join = torch.cuda.Event()
            join.record(st)
            main.wait_event(join)

    s0 = 3 * w.d
    cycles = graph_cycles(args, w.R)
    graphs = PhaseGraphs(torch, step, w.R, s0, cycle_fn=cycle, cycles=cycles)
    graphs.run(0, args.warmup)
    torch.cuda.synchronize()
    # fresh host data and a cleared output block: the checks below prove that the
    # graphs carry both copies
    host_in[off_w:].view(torch.float32).normal_()
    host_out.zero_()
    win_ms, n_win, _ = steady_windows(torch, graphs.run, args.steps, args.warmup)
    ms = win_ms / args.steps
    w.check_status()
    last = args.warmup + args.steps * (n_win + 1) - 1          # the last step replayed
    s_last = s0 + last % w.R
    assert torch.equal(dev_in[(s_last + 1) % NB].cpu(), host_in), "input copy missing from the step graph"
    assert torch.equal(host_out, dev_out[(s_last - 1) % NB].cpu()) and bool(host_out.any()), \
        "output copy missing from the step graph"
    return {"value": B * 4 / (ms / 1e3), "unit": UNIT, "ms_per_step": ms, "h2d_bytes_per_step": in_bytes,
            "d2h_bytes_per_step": out_bytes,
            "launch": f"CUDA graphs of {w.R * cycles} consecutive steps with only the data's "
            f"dependencies between them; {NB} staging buffers; per step the next step's "
            "input copy and the previous step's output copy on two copy streams, overlapped with 4 window-row "
            "placements and 4 layer calls in parallel branches"}


# ------------------------------------------------------------------ other configurations
# The remaining workload configurations, one JSON line each (--workload):
#   full131k   decode Full mode on a decoder source layer (m=1): batch 64 x
#              131,072 entries, one query per sequence at t = N-1
#   prefill8k  prefill chunk on an encoder source layer (m=2): 8192 queries at
#              t = 131,072..139,263 over 69,632 entries, causal
#   cachewrite cache write of 4 source layers (3 at m=2, 1 at m=1) over
#              1,048,576 tokens each
#   hisa131k   HISA decode (block-mean first stage, Reindex second stage) on
#              the full131k cache, the HSI Full call timed beside it
#   hisa1m     the same at batch 16 x 1,048,576 entries
FP4_PER_BF16 = 13.5 / 2.25          # nominal dense fp4 : bf16 tensor ratio
FP32_FMA_PER_SM_CLK = 128           # fp32 FMA lanes per SM and clock


def _weights(torch, seed):
    import numpy as np
    import synth
    g = synth.rng(seed)
    w0, w1 = synth.compressor_weights(g)
    W = synth.index_projection(g)
    return (torch.from_numpy(w0).cuda(), torch.from_numpy(w1).cuda(),
            torch.from_numpy(np.ascontiguousarray(W).view(np.int16)).cuda())


def _write_cache(csa2, torch, cache, T, seed, wts, rope, ws, chunk=1 << 17):
    """Cache write of every sequence's T tokens of seeded N(0,1) latents."""
    import synth
    w0, w1, w_idx = wts
    for b in range(cache.B):
        view = cache.sequence(b)
        for c0 in range(0, T, chunk):
            n = min(chunk, T - c0)
            x = synth.torch_latents(seed * 100_003 + b * 1_009 + c0 // chunk, (1, n), "cuda")
            start = torch.tensor([c0 // cache.m], dtype=torch.int64, device="cuda")
            csa2.compress_quantize(view, x.view(torch.int16), start, w0, w1, rope, w_idx, ws)


def _events_ms(torch, fn, steps, flush=None):
    """Device time of `steps` calls of fn.  With `flush`, every call runs after an
    L2 flush and is timed alone (the flushes are outside the timed regions)."""
    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps
    total = 0.0
    for i in range(steps):
        flush.fill_(i & 255)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        total += e0.elapsed_time(e1)
    return total / steps


def _line(args, world, metric, unit, value, ms, dtype, config, roofline, extra):
    line = {"metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": dtype, "data": "synthetic", "config": config, "roofline": roofline,
            "cpu_baseline": None, "e2e": None}
    line.update(extra)
    return line


def run_full131k(args, torch, csa2):
    """Decode Full mode: index scan of every visible entry, block top-2048,
    top-512, attention; batch 64 x 131,072 entries (2.99 GB of cache, > L2)."""
    import synth
    rank, world, local = dist_info()
    B, N, dev = 64, 1 << 17, "cuda"
    cache = csa2.Cache(B, N, 1, device=dev)
    wts = _weights(torch, 2)
    ones = torch.ones(D, device=dev)
    rope = csa2.rope_table(N).to(dev)
    ws_cw = csa2.Workspace(1 << 16, device=dev)
    _write_cache(csa2, torch, cache, N, 2, (ones, ones, wts[2]), rope, ws_cw)
    cache.n_entries.fill_(N)
    assert ws_cw.sync_status()[0] == 0
    del rope
    q_pos = torch.full((B, 1), N - 1, dtype=torch.int64, device=dev)
    swa_base = torch.full((B,), N - WIN, dtype=torch.int64, device=dev)
    q_idx = synth.torch_normal(21, (B, 1, HI, DI), torch.bfloat16, dev)
    w_head = synth.torch_normal(22, (B, 1, HI), torch.float32, dev)
    q = synth.torch_normal(23, (B, 1, H, D), torch.bfloat16, dev)
    swa = synth.torch_swa_rows(24, (B, WIN), dev)
    pool = torch.empty((B, 1, M_BLK), dtype=torch.int32, device=dev)
    sel = torch.empty((B, 1, K_SEL), dtype=torch.int32, device=dev)
    out = torch.empty((B, 1, H, D), dtype=torch.bfloat16, device=dev)
    ws = csa2.Workspace(csa2.decode_workspace_size(csa2.MODE_FULL, B, 1, N, M_BLK, K_SEL), device=dev)
    split = latency_split(torch, B, 1)

    def step():
        csa2.decode(csa2.MODE_FULL, cache, q_pos=q_pos, q=q.view(torch.int16), swa=swa.view(torch.int16),
                    swa_base_pos=swa_base, scale=1 / math.sqrt(D), sel=sel, out=out.view(torch.int16), ws=ws,
                    M=M_BLK, max_n=N, q_idx=q_idx.view(torch.int16), w_head=w_head, pool_blocks=pool,
                    attn_split=split)
    graph = _capture(torch, step)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    with ClockSampler(local) as clk:
        ms = _events_ms(torch, graph.replay, args.steps)
    ms = max_over_ranks(ms, world)
    assert ws.sync_status()[0] == 0
    # the dominant kernel alone: the index scan (public call, same inputs)
    scores = torch.empty((B, 1, N), dtype=torch.float32, device=dev)
    ws_s = csa2.Workspace(1 << 16, device=dev)
    g_s = _capture(torch, lambda: csa2.index_score(cache, q_idx.view(torch.int16), w_head, q_pos, scores, N, ws_s))
    g_s.replay()
    scan_ms = _events_ms(torch, g_s.replay, max(args.steps, 20))
    cpu = None
    if args.cpu_sample_queries > 0:
        n_q = max(1, args.cpu_sample_queries // 24)
        dt = OracleLayer(N, 1).run([N - 1] * n_q)
        cpu = _oracle_line(n_q / dt, "query-tokens/s", f"{n_q} Full-mode queries over {N:,} entries (m=1) on a "
                                                       f"cache of random stored bytes, {dt:.1f} s")
    hbm, _, which = peaks()
    scan_bytes = B * N * (IDX_ENTRY + 4) + B * (HI * DI * 2 + HI * 4)       # index K read + scores written
    per_query = N * IDX_ENTRY + HI * DI * 2 + HI * 4 + ATTN_BYTES + M_BLK * 4 + K_SEL * 4
    achieved = scan_bytes / (scan_ms / 1e3) / 1e9
    return _line(args, world, "CSA2 Full decode query-tokens/s/layer at 131K ctx, batch 64", "query-tokens/s",
                 B * world / (ms / 1e3), ms, "fp4-e2m1 cache, mxfp4 index, f16 mma fp32 acc",
                 {"workload": "decode Full mode, m=1, 64 sequences x 131,072 entries, one query each",
                  "M_blocks": M_BLK, "K": K_SEL, "window": WIN,
                  "l2": "inputs larger than L2 (2.99 GB of cache; the scan reads 570 MB per step)",
                  "launch": "one CUDA graph per step (index scan, block and entry selection, attention)",
                  "attention": f"{split} CTAs per query (the key chunks split, partial softmax states merged)"},
                 {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                  "traffic": ncu_traffic("index_score_tc_kernel<1>"), "kernel": "index_score_tc_kernel<1>",
                  "algorithmic_bytes_per_launch": scan_bytes, "avg_launch_ms": scan_ms, "peak_source": which},
                 {"step_hbm": {"algorithmic_bytes": B * per_query, "GB_s": B * per_query / (ms / 1e3) / 1e9,
                               "frac": B * per_query / (ms / 1e3) / 1e9 / hbm},
                  "clocks": clk.summary(), "gpu_launches": args.steps * 5, "cpu_baseline": cpu})


def _hisa_workload(args, torch, csa2, B, N, seed):
    """HISA decode on a decoder source layer (m = 1), one query per sequence at
    t = N - 1: the newest block's summary update, the first stage (summary
    scan and top-2048 blocks) and the Reindex second stage with attention.
    The HSI Full call on the same cache and queries is timed beside it."""
    import synth
    rank, world, local = dist_info()
    dev = "cuda"
    cache = csa2.Cache(B, N, 1, device=dev)
    wts = _weights(torch, seed)
    ones = torch.ones(D, device=dev)
    rope = csa2.rope_table(N).to(dev)
    ws_cw = csa2.Workspace(1 << 16, device=dev)
    _write_cache(csa2, torch, cache, N, seed, (ones, ones, wts[2]), rope, ws_cw)
    cache.n_entries.fill_(N)
    assert ws_cw.sync_status()[0] == 0
    del rope
    nb = -(-N // 8)
    store = csa2.BlockSummaries(cache, device=dev)
    first0 = torch.zeros(B, dtype=torch.int64, device=dev)
    build_ms = _events_ms(torch, lambda: csa2.block_summary(cache, store, first0, nb, ws_cw), 3)
    q_pos = torch.full((B, 1), N - 1, dtype=torch.int64, device=dev)
    newest = torch.full((B,), (N - 1) // 8, dtype=torch.int64, device=dev)
    swa_base = torch.full((B,), N - WIN, dtype=torch.int64, device=dev)
    q_idx = synth.torch_normal(seed * 10 + 1, (B, 1, HI, DI), torch.bfloat16, dev)
    w_head = synth.torch_normal(seed * 10 + 2, (B, 1, HI), torch.float32, dev)
    q = synth.torch_normal(seed * 10 + 3, (B, 1, H, D), torch.bfloat16, dev)
    swa = synth.torch_swa_rows(seed * 10 + 4, (B, WIN), dev)
    pool = torch.empty((B, 1, M_BLK), dtype=torch.int32, device=dev)
    sel = torch.empty((B, 1, K_SEL), dtype=torch.int32, device=dev)
    out = torch.empty((B, 1, H, D), dtype=torch.bfloat16, device=dev)
    ws_s = csa2.Workspace(1 << 16, device=dev)
    ws_h = csa2.Workspace(csa2.hisa_blocks_workspace_size(B, 1, N), device=dev)
    ws_r = csa2.Workspace(csa2.decode_workspace_size(csa2.MODE_REINDEX, B, 1, N, M_BLK, K_SEL), device=dev)
    split = latency_split(torch, B, 1)
    common = dict(q_pos=q_pos, q=q.view(torch.int16), swa=swa.view(torch.int16), swa_base_pos=swa_base,
                  scale=1 / math.sqrt(D), sel=sel, out=out.view(torch.int16), M=M_BLK, max_n=N,
                  q_idx=q_idx.view(torch.int16), w_head=w_head, pool_blocks=pool, attn_split=split)

    def summary():
        csa2.block_summary(cache, store, newest, 1, ws_s)

    def stage1():
        csa2.hisa_blocks(cache, store, q_idx.view(torch.int16), w_head, q_pos, N, M_BLK, pool, ws_h)

    def stage2():
        csa2.decode(csa2.MODE_REINDEX, cache, ws=ws_r, **common)

    graph = _capture(torch, lambda: (summary(), stage1(), stage2()))
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    with ClockSampler(local) as clk:
        ms = _events_ms(torch, graph.replay, args.steps)
    ms = max_over_ranks(ms, world)
    for w in (ws_s, ws_h, ws_r):
        assert w.sync_status()[0] == 0
    reps = max(args.steps, 20)
    parts = {}
    for name, fn in (("summary_update", summary), ("stage1_blocks", stage1), ("stage2_reindex", stage2)):
        g = _capture(torch, fn)
        parts[name] = _graph_ms(torch, g, reps)
    # the HSI Full call on the same cache and query, for comparison
    ws_f = csa2.Workspace(csa2.decode_workspace_size(csa2.MODE_FULL, B, 1, N, M_BLK, K_SEL), device=dev)
    g_full = _capture(torch, lambda: csa2.decode(csa2.MODE_FULL, cache, ws=ws_f, **common))
    full_ms = _graph_ms(torch, g_full, reps)
    # pool recall: the share of the Full call's top-512 (the exact top-K over
    # every visible entry) whose block is in the HISA pool, and in the HSI pool
    sel_f, pool_f = torch.empty_like(sel), torch.empty_like(pool)
    csa2.decode(csa2.MODE_FULL, cache, ws=ws_f, **dict(common, sel=sel_f, pool_blocks=pool_f))
    stage1()
    torch.cuda.synchronize()
    recall = {}
    for name, pb in (("hisa", pool), ("hsi", pool_f)):
        hit = tot = 0
        for b in range(B):
            ids = sel_f[b, 0][sel_f[b, 0] >= 0]
            hit += int(torch.isin(torch.div(ids, 8, rounding_mode="floor"), pb[b, 0]).sum())
            tot += int(ids.numel())
        recall[name] = hit / max(tot, 1)
    # the summary scan alone: the index scan over the summary store read as a
    # cache of nb rows (the view hisa_blocks builds on the device)
    view = csa2.Cache.__new__(csa2.Cache)
    view.B, view.cap, view.m = B, store.sum_cap, 1
    view.main_kv, view.idx_codes, view.idx_scales = cache.main_kv, store.codes, store.scales
    view.n_entries = torch.full((B,), nb, dtype=torch.int32, device=dev)
    view_pos = torch.full((B, 1), nb - 1, dtype=torch.int64, device=dev)
    scores = torch.empty((B, 1, nb), dtype=torch.float32, device=dev)
    g_scan = _capture(torch, lambda: csa2.index_score(view, q_idx.view(torch.int16), w_head, view_pos, scores, nb,
                                                      ws_s))
    scan_ms = _graph_ms(torch, g_scan, reps)
    assert ws_s.sync_status()[0] == 0
    cpu = None
    if args.cpu_sample_queries > 0:
        # about 10 s of oracle work at 131,072 entries (the first stage grows with N)
        n_q = max(1, min(args.cpu_sample_queries, 400 * (1 << 17) // N))
        cpu_v, cpu_dt = OracleHisa(N).run(n_q)
        cpu = {"value": cpu_v, "unit": "query-tokens/s", "cores": oracle_threads(), "kind": "oracle",
               "sample": f"{n_q} queries over {N:,} entries (newest-block summary, first stage over "
                         f"{nb:,} summary rows, Reindex over {M_BLK} blocks, attention), {cpu_dt:.1f} s"}
    hbm, _, which = peaks()
    scan_bytes = B * nb * (IDX_ENTRY + 4) + B * (HI * DI * 2 + HI * 4)
    achieved = scan_bytes / (scan_ms / 1e3) / 1e9
    per_query = (8 * IDX_ENTRY + IDX_ENTRY) + nb * (IDX_ENTRY + 4 + 4) + M_BLK * 4 + REINDEX_BYTES
    kname = "index_score_tc_kernel<1>"
    return _line(args, world, f"CSA2 HISA decode query-tokens/s/layer at {N // 1024}K ctx, batch {B}",
                 "query-tokens/s", B * world / (ms / 1e3), ms, "fp4-e2m1 cache, mxfp4 index, f16 mma fp32 acc",
                 {"workload": f"HISA decode, m=1, {B} sequences x {N:,} entries, one query each: newest block "
                              f"summary, top-{M_BLK} blocks by mean-key score, Reindex top-{K_SEL} over them, "
                              f"attention",
                  "M_blocks": M_BLK, "K": K_SEL, "window": WIN,
                  "l2": "inputs larger than L2 (the summary store and cache exceed 129 MB)",
                  "launch": "one CUDA graph per step (summary update, view, summary scan, block selection, "
                            "Reindex scan+select, attention)",
                  "attention": f"{split} CTAs per query (the key chunks split, partial softmax states merged)"},
                 {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                  "traffic": ncu_traffic(f"{kname}:summaries_{B}x{nb}"), "kernel": kname + " over the summary store",
                  "algorithmic_bytes_per_launch": scan_bytes, "avg_launch_ms": scan_ms, "peak_source": which},
                 {"parts_ms": parts, "hsi_full_call_ms": full_ms, "summary_build_ms": build_ms,
                  "pool_recall_of_exact_top512": recall, "cpu_baseline": cpu,
                  "step_hbm": {"algorithmic_bytes": B * per_query, "GB_s": B * per_query / (ms / 1e3) / 1e9,
                               "frac": B * per_query / (ms / 1e3) / 1e9 / hbm},
                  "clocks": clk.summary(),
                  # summary, view, scan, 3 selection kernels (rows over 4,096 blocks), Reindex, attention
                  "gpu_launches": args.steps * 8})


def run_hisa131k(args, torch, csa2):
    return _hisa_workload(args, torch, csa2, 64, 1 << 17, 2)


def run_hisa1m(args, torch, csa2):
    return _hisa_workload(args, torch, csa2, 16, 1 << 20, 3)


def run_decoder1m(args, torch, csa2):
    """One token through a whole decoder at 1M entries, batch 16: the source
    layer in Full mode + 3 Reuse layers, then 4 x (Reindex + 3 Reuse) on the
    same cache (1 Full scan, 4 Reindexes and 15 Reuses per token); each
    Full/Reindex call packs its selection for its 3 Reuse layers.  One CUDA
    graph per token, calls in order on one stream."""
    import synth
    rank, world, local = dist_info()
    B, N, dev = 16, args.seq_len, "cuda"
    cache = csa2.Cache(B, N, 1, device=dev)
    ones = torch.ones(D, device=dev)
    wts = _weights(torch, 3)
    rope = csa2.rope_table(N).to(dev)
    ws_cw = csa2.Workspace(1 << 16, device=dev)
    _write_cache(csa2, torch, cache, N, 3, (ones, ones, wts[2]), rope, ws_cw)
    cache.n_entries.fill_(N)
    assert ws_cw.sync_status()[0] == 0
    del rope
    q_pos = torch.full((B, 1), N - 1, dtype=torch.int64, device=dev)
    swa_base = torch.full((B,), N - WIN, dtype=torch.int64, device=dev)
    n_layers, groups = 20, 5                      # layer 4g is Full (g = 0) or Reindex, then 3 Reuse
    qs = [synth.torch_normal(300 + l, (B, 1, H, D), torch.bfloat16, dev) for l in range(n_layers)]
    swas = [synth.torch_swa_rows(400 + l, (B, WIN), dev) for l in range(n_layers)]
    q_idx = [synth.torch_normal(500 + g, (B, 1, HI, DI), torch.bfloat16, dev) for g in range(groups)]
    w_head = [synth.torch_normal(600 + g, (B, 1, HI), torch.float32, dev) for g in range(groups)]
    pool = torch.empty((B, 1, M_BLK), dtype=torch.int32, device=dev)
    sels = [torch.empty((B, 1, K_SEL), dtype=torch.int32, device=dev) for _ in range(groups)]
    packs = [torch.empty((B, 1, K_SEL, MAIN_ENTRY), dtype=torch.uint8, device=dev) for _ in range(groups)]
    outs = [torch.empty((B, 1, H, D), dtype=torch.bfloat16, device=dev) for _ in range(n_layers)]
    modes = [csa2.MODE_FULL, csa2.MODE_REINDEX, csa2.MODE_REUSE]
    wss = {m: csa2.Workspace(csa2.decode_workspace_size(m, B, 1, N, M_BLK, K_SEL), device=dev) for m in modes}
    split = latency_split(torch, B, 1)

    def step():
        for l in range(n_layers):
            g, k = divmod(l, 4)
            mode = csa2.MODE_REUSE if k else (csa2.MODE_FULL if g == 0 else csa2.MODE_REINDEX)
            csa2.decode(mode, cache, q_pos=q_pos, q=qs[l].view(torch.int16), swa=swas[l].view(torch.int16),
                        swa_base_pos=swa_base, scale=1 / math.sqrt(D), sel=sels[g], out=outs[l].view(torch.int16),
                        ws=wss[mode], M=M_BLK, max_n=N, q_idx=q_idx[g].view(torch.int16), w_head=w_head[g],
                        pool_blocks=pool, packed_sel=packs[g], attn_split=split)
    graph = _capture(torch, step)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    with ClockSampler(local) as clk:
        ms = _events_ms(torch, graph.replay, args.steps)
    ms = max_over_ranks(ms, world)
    for w in wss.values():
        assert w.sync_status()[0] == 0
    # the dominant kernel alone: the Full layer's index scan over 16 x N entries
    scores = torch.empty((B, 1, N), dtype=torch.float32, device=dev)
    ws_s = csa2.Workspace(1 << 16, device=dev)
    g_s = _capture(torch, lambda: csa2.index_score(cache, q_idx[0].view(torch.int16), w_head[0], q_pos, scores,
                                                   N, ws_s))
    g_s.replay()
    scan_ms = _events_ms(torch, g_s.replay, max(args.steps, 20))
    hbm, _, which = peaks()
    scan_bytes = B * N * (IDX_ENTRY + 4) + B * (HI * DI * 2 + HI * 4)
    full_q = N * IDX_ENTRY + HI * DI * 2 + HI * 4 + ATTN_BYTES + M_BLK * 4 + K_SEL * 4 + K_SEL * MAIN_ENTRY
    per_query = full_q + 4 * REINDEX_BYTES + 15 * REUSE_BYTES
    achieved = scan_bytes / (scan_ms / 1e3) / 1e9
    return _line(args, world, "CSA2 whole-decoder query-token-layers/s at 1M ctx (Full + 3 Reuse, 4 x (Reindex + "
                 "3 Reuse)), batch 16", UNIT, B * n_layers * world / (ms / 1e3), ms,
                 "fp4-e2m1 cache, mxfp4 index, f16 mma fp32 acc",
                 {"workload": f"one token through a 20-layer decoder block chain, {N:,} entries/seq, batch 16: "
                              "Full source layer + 3 Reuse, then 4 x (Reindex on the Full layer's pool + 3 Reuse), "
                              "one cache", "global_batch": B, "seq_len": N, "M_blocks": M_BLK, "K": K_SEL,
                  "window": WIN,
                  "l2": "the Full scan reads the 1.1 GB of index K every token (larger than L2); the Reindex layers "
                        "share the Full layer's pool",
                  "selection": "each Full/Reindex call packs its selected entries for its 3 Reuse calls",
                  "launch": "one CUDA graph per token, the 20 calls in order on one stream",
                  "attention": f"{split} CTAs per query (the key chunks split, partial softmax states merged)"},
                 {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                  "traffic": None, "kernel": "index_score_tc_kernel<1> (Full layer at 1M)",
                  "algorithmic_bytes_per_launch": scan_bytes, "avg_launch_ms": scan_ms, "peak_source": which},
                 {"step_hbm": {"algorithmic_bytes": B * per_query, "GB_s": B * per_query / (ms / 1e3) / 1e9,
                               "frac": B * per_query / (ms / 1e3) / 1e9 / hbm},
                  "ms_per_token": ms, "clocks": clk.summary(), "cpu_baseline": _decoder_oracle(args, N),
                  "gpu_launches": args.steps * (5 + 4 * 2 + 15)})   # Full 5, Reindex 2, Reuse 1


def run_prefill8k(args, torch, csa2):
    """Prefill chunk: 8192 causal queries, one Full-mode call (index scan of
    5 queries per CTA, per-query block top-2048 and top-512, attention)."""
    import synth
    rank, world, local = dist_info()
    m, P, C, dev = 2, 131072, 8192, "cuda"
    T = P + C
    N = T // m
    cache = csa2.Cache(1, N, m, device=dev)
    wts = _weights(torch, 4)
    rope = csa2.rope_table(N).to(dev)
    ws_cw = csa2.Workspace(1 << 16, device=dev)
    _write_cache(csa2, torch, cache, T, 4, wts, rope, ws_cw)
    cache.n_entries.fill_(N)
    assert ws_cw.sync_status()[0] == 0
    Q = C
    q_pos = torch.arange(P, T, dtype=torch.int64, device=dev)[None]
    swa_base = torch.full((1,), P - (WIN - 1), dtype=torch.int64, device=dev)
    q_idx = synth.torch_normal(41, (1, Q, HI, DI), torch.bfloat16, dev)
    w_head = synth.torch_normal(42, (1, Q, HI), torch.float32, dev)
    q = synth.torch_normal(43, (1, Q, H, D), torch.bfloat16, dev)
    swa = synth.torch_swa_rows(44, (1, Q + WIN - 1), dev)
    pool = torch.empty((1, Q, M_BLK), dtype=torch.int32, device=dev)
    sel = torch.empty((1, Q, K_SEL), dtype=torch.int32, device=dev)
    out = torch.empty((1, Q, H, D), dtype=torch.bfloat16, device=dev)
    ws = csa2.Workspace(csa2.decode_workspace_size(csa2.MODE_FULL, 1, Q, N, M_BLK, K_SEL), device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        csa2.decode(csa2.MODE_FULL, cache, q_pos=q_pos, q=q.view(torch.int16), swa=swa.view(torch.int16),
                    swa_base_pos=swa_base, scale=1 / math.sqrt(D), sel=sel, out=out.view(torch.int16), ws=ws,
                    M=M_BLK, max_n=N, q_idx=q_idx.view(torch.int16), w_head=w_head, pool_blocks=pool)
    graph = _capture(torch, step)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    with ClockSampler(local) as clk:
        ms = _events_ms(torch, graph.replay, args.steps, flush=flush)
    ms = max_over_ranks(ms, world)
    assert ws.sync_status()[0] == 0
    # the tensor-core kernel alone: the grouped index scan (public call, same inputs)
    scores = torch.empty((1, Q, N), dtype=torch.float32, device=dev)
    ws_s = csa2.Workspace(1 << 16, device=dev)
    g_s = _capture(torch, lambda: csa2.index_score(cache, q_idx.view(torch.int16), w_head, q_pos, scores, N, ws_s))
    g_s.replay()
    scan_ms = _events_ms(torch, g_s.replay, max(args.steps, 10), flush=flush)
    _, bf16, which = peaks()
    pairs = sum(min((t + 1) // m, N) for t in range(P, T))                  # (query, visible entry) pairs
    flops = pairs * HI * DI * 2
    fp4_peak = bf16 * FP4_PER_BF16
    achieved = flops / (scan_ms / 1e3) / 1e12
    return _line(args, world, "CSA2 prefill-chunk query-tokens/s, 8192 new tokens on a 131K prefix",
                 "query-tokens/s", Q * world / (ms / 1e3), ms, "fp4-e2m1 cache, mxfp4 index, f16 mma fp32 acc",
                 {"workload": "prefill chunk, m=2, 131,072-token prefix + 8192 new tokens (69,632 entries), "
                              "8192 causal queries, batch 1",
                  "M_blocks": M_BLK, "K": K_SEL, "window": WIN,
                  "l2": "L2 flushed (256 MB write) before every timed step; the caches (24 MB) fit in L2",
                  "launch": "one CUDA graph per step"},
                 {"bound": "tensor", "achieved": achieved, "peak": fp4_peak, "unit": "TFLOP/s",
                  "frac": achieved / fp4_peak, "traffic": None, "kernel": "index_score_tc_kernel<5>",
                  "algorithmic_flops_per_launch": flops, "avg_launch_ms": scan_ms,
                  "peak_source": f"{which} bf16 x {FP4_PER_BF16:g} (nominal fp4:bf16 dense ratio)"},
                 {"clocks": clk.summary(), "gpu_launches": args.steps * 5,
                  "cpu_baseline": _prefill_oracle(args, P, T, N, m, 0)})


def run_prefillblock(args, torch, csa2):
    """An encoder block over the prefill chunk: the source layer (m=2) in Full
    mode + 5 Reuse layers with fresh queries and windows, reading the Full
    layer's selection from the same (L2-resident) cache.  One CUDA graph per
    chunk, L2 flushed before each."""
    import synth
    rank, world, local = dist_info()
    m, P, C, dev = 2, 131072, 8192, "cuda"
    T = P + C
    N = T // m
    cache = csa2.Cache(1, N, m, device=dev)
    wts = _weights(torch, 4)
    rope = csa2.rope_table(N).to(dev)
    ws_cw = csa2.Workspace(1 << 16, device=dev)
    _write_cache(csa2, torch, cache, T, 4, wts, rope, ws_cw)
    cache.n_entries.fill_(N)
    assert ws_cw.sync_status()[0] == 0
    Q, n_layers = C, 6
    q_pos = torch.arange(P, T, dtype=torch.int64, device=dev)[None]
    swa_base = torch.full((1,), P - (WIN - 1), dtype=torch.int64, device=dev)
    q_idx = synth.torch_normal(41, (1, Q, HI, DI), torch.bfloat16, dev)
    w_head = synth.torch_normal(42, (1, Q, HI), torch.float32, dev)
    qs = [synth.torch_normal(700 + l, (1, Q, H, D), torch.bfloat16, dev) for l in range(n_layers)]
    swas = [synth.torch_swa_rows(800 + l, (1, Q + WIN - 1), dev) for l in range(n_layers)]
    pool = torch.empty((1, Q, M_BLK), dtype=torch.int32, device=dev)
    sel = torch.empty((1, Q, K_SEL), dtype=torch.int32, device=dev)
    outs = [torch.empty((1, Q, H, D), dtype=torch.bfloat16, device=dev) for _ in range(n_layers)]
    ws_f = csa2.Workspace(csa2.decode_workspace_size(csa2.MODE_FULL, 1, Q, N, M_BLK, K_SEL), device=dev)
    ws_r = csa2.Workspace(csa2.decode_workspace_size(csa2.MODE_REUSE, 1, Q, N, M_BLK, K_SEL), device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        for l in range(n_layers):
            csa2.decode(csa2.MODE_FULL if l == 0 else csa2.MODE_REUSE, cache, q_pos=q_pos,
                        q=qs[l].view(torch.int16), swa=swas[l].view(torch.int16), swa_base_pos=swa_base,
                        scale=1 / math.sqrt(D), sel=sel, out=outs[l].view(torch.int16), ws=ws_f if l == 0 else ws_r,
                        M=M_BLK, max_n=N, q_idx=q_idx.view(torch.int16), w_head=w_head, pool_blocks=pool)
    graph = _capture(torch, step)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    with ClockSampler(local) as clk:
        ms = _events_ms(torch, graph.replay, args.steps, flush=flush)
    ms = max_over_ranks(ms, world)
    assert ws_f.sync_status()[0] == 0 and ws_r.sync_status()[0] == 0
    # the tensor-bound kernel alone: the grouped index scan
    scores = torch.empty((1, Q, N), dtype=torch.float32, device=dev)
    ws_s = csa2.Workspace(1 << 16, device=dev)
    g_s = _capture(torch, lambda: csa2.index_score(cache, q_idx.view(torch.int16), w_head, q_pos, scores, N, ws_s))
    g_s.replay()
    scan_ms = _events_ms(torch, g_s.replay, max(args.steps, 10), flush=flush)
    _, bf16, which = peaks()
    pairs = sum(min((t + 1) // m, N) for t in range(P, T))
    flops = pairs * HI * DI * 2
    fp4_peak = bf16 * FP4_PER_BF16
    achieved = flops / (scan_ms / 1e3) / 1e12
    attn_flops = n_layers * Q * (K_SEL + WIN) * H * D * 4
    return _line(args, world, "CSA2 encoder-block prefill query-token-layers/s (Full + 5 Reuse), 8192 new tokens "
                 "on a 131K prefix", UNIT, Q * n_layers * world / (ms / 1e3), ms,
                 "fp4-e2m1 cache, mxfp4 index, f16 mma fp32 acc",
                 {"workload": "encoder block on a prefill chunk, m=2, 131,072-token prefix + 8192 new tokens "
                              "(69,632 entries): the Full source layer + 5 Reuse layers (fresh queries and windows) "
                              "on its selection, batch 1",
                  "M_blocks": M_BLK, "K": K_SEL, "window": WIN,
                  "l2": "L2 flushed (256 MB write) before every timed chunk; the caches (24 MB) fit in L2",
                  "selection": "the Reuse layers gather from the L2-resident cache (no packed copy)",
                  "launch": "one CUDA graph per chunk, the 6 calls in order"},
                 {"bound": "tensor", "achieved": achieved, "peak": bf16 * FP4_PER_BF16, "unit": "TFLOP/s",
                  "frac": achieved / fp4_peak, "traffic": None, "kernel": "index_score_tc_kernel<5>",
                  "algorithmic_flops_per_launch": flops, "avg_launch_ms": scan_ms,
                  "peak_source": f"{which} bf16 x {FP4_PER_BF16:g} (nominal fp4:bf16 dense ratio)"},
                 {"attention_bf16_flops_per_chunk": attn_flops, "clocks": clk.summary(),
                  "cpu_baseline": _prefill_oracle(args, P, T, N, m, 5),
                  "gpu_launches": args.steps * (5 + 5)})   # Full: scan, 3 selection, attention; Reuse: attention


def run_cachewrite(args, torch, csa2):
    """Cache write of 4 source layers (3 at m=2, 1 at m=1) over 1,048,576 tokens:
    compressor, RMSNorm, RoPE, E2M1 + E4M3 main KV, index-K projection + MXFP4."""
    import synth
    rank, world, local = dist_info()
    T, dev = 1 << 20, "cuda"
    wts = _weights(torch, 1)
    rope = csa2.rope_table(T).to(dev)
    ws = csa2.Workspace(1 << 16, device=dev)
    layers = []
    for layer, m in enumerate((2, 2, 2, 1)):
        x = synth.torch_latents(10 + layer, (1, T), dev)                      # 1 GiB of bf16 latents each
        layers.append((csa2.Cache(1, T // m, m, device=dev), x))
    start = torch.zeros((1,), dtype=torch.int64, device=dev)

    def step():
        for cache, x in layers:
            csa2.compress_quantize(cache, x.view(torch.int16), start, wts[0], wts[1], rope, wts[2], ws)
    graph = _capture(torch, step)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    with ClockSampler(local) as clk:
        ms = _events_ms(torch, graph.replay, args.steps)
    ms = max_over_ranks(ms, world)
    assert ws.sync_status()[0] == 0
    entries = sum(T // m for m in (2, 2, 2, 1))
    out_bytes = sum(c.main_kv.numel() + c.idx_codes.numel() + c.idx_scales.numel() for c, _ in layers)
    assert out_bytes == 890 * T
    fma = entries * DI * D                                                 # the index-K projection
    clocks = clk.summary()
    props = torch.cuda.get_device_properties(0)
    sm_mhz = clocks.get("sm_max_mhz") or 2070.0
    fma_peak = props.multi_processor_count * FP32_FMA_PER_SM_CLK * sm_mhz * 1e6
    achieved = fma / (ms / 1e3)
    hbm, _, which = peaks()
    bytes_step = 4 * T * D * 2 + out_bytes
    return _line(args, world, "CSA2 cache-write tokens/s (4 source layers x 1M tokens)", "tokens/s",
                 4 * T * world / (ms / 1e3), ms, "bf16 in, fp32 math, fp4/fp8 codes out",
                 {"workload": "cache write, 4 source layers (3 at m=2, 1 at m=1) x 1,048,576 tokens, 890 B/token out",
                  "l2": "inputs larger than L2 (4 GiB of latents per step)", "launch": "one CUDA graph per step"},
                 {"bound": "alu", "achieved": achieved / 1e12, "peak": fma_peak / 1e12, "unit": "TFMA/s",
                  "frac": achieved / fma_peak, "traffic": None, "kernel": "cache_write_kernel",
                  "algorithmic_fma_per_step": fma, "avg_launch_ms": ms / 4,
                  "peak_source": f"{props.multi_processor_count} SMs x {FP32_FMA_PER_SM_CLK} fp32 FMA/clk x "
                                 f"{sm_mhz:.0f} MHz"},
                 {"step_hbm": {"algorithmic_bytes": bytes_step, "GB_s": bytes_step / (ms / 1e3) / 1e9,
                               "frac": bytes_step / (ms / 1e3) / 1e9 / hbm},
                  "clocks": clocks, "gpu_launches": args.steps * 4, "cpu_baseline": _cachewrite_oracle(args)})


# ------------------------------------------------------------------ CPU oracle sample
class OracleChain:
    """Oracle (binary64 numpy + C cache write) on the per-query work of the
    decode step: Reindex (score a 16,384-entry pool, top-512, attention) and
    three Reuse attentions.  The pool's entries are written by the oracle's own
    cache write during set-up (untimed); entry ids are compacted so the pool is
    blocks 0..2047, which leaves the per-query work unchanged."""

    def __init__(self, seed: int = 9, n_query_sets: int = 8, swa_fp8: bool = False):
        import numpy as np
        import oracle
        import synth
        self.oracle = oracle
        g = synth.rng(seed)
        self.n = M_BLK * 8
        x = synth.latents(g, self.n)
        w0, w1 = synth.compressor_weights(g)
        W = synth.index_projection(g)
        self.main, self.codes, self.scales = oracle.compress_quantize(x, 1, w0, w1, W)
        self.swa = synth.swa_rows(g, WIN)
        if swa_fp8:                  # E4M3 window rows (quantised untimed, as the GPU leg does)
            self.swa = oracle.swa_fp8_quantize(self.swa)
        self.pool = np.arange(M_BLK, dtype=np.int32)
        self.qs = [(synth.index_queries(g), synth.head_weights(g), [synth.main_queries(g) for _ in range(4)])
                   for _ in range(n_query_sets)]

    def run(self, n_queries: int) -> tuple[float, float]:
        o = self.oracle
        common = dict(t=self.n - 1, m=1, n_entries=self.n, main_kv=self.main, idx_codes=self.codes,
                      idx_scales=self.scales, swa=self.swa, swa_base=self.n - WIN, scale=1 / math.sqrt(D),
                      M=M_BLK, K=K_SEL)
        t0 = time.perf_counter()
        for i in range(n_queries):
            q_idx, wh, q4 = self.qs[i % len(self.qs)]
            _, sel, _ = o.decode_query(o.REINDEX, q=q4[0], q_idx=q_idx, w_head=wh, pool_blocks=self.pool, **common)
            for layer in range(1, 4):
                o.decode_query(o.REUSE, q=q4[layer], sel=sel, **common)
        dt = time.perf_counter() - t0
        return n_queries * 4 / dt, dt


class OracleHisa:
    """Oracle on the per-query work of a HISA decode step over n entries: the
    newest block's summary, the first stage over all ceil(n/8) summary rows,
    the Reindex second stage over the chosen blocks and the attention.  The
    cache is stored bytes drawn at random (index keys: synth.index_key_bytes;
    main entries: uniform codes with E4M3 scales in [0.5, 1]), the summary
    store is built once untimed."""

    def __init__(self, n: int, seed: int = 11, n_query_sets: int = 4):
        import numpy as np
        import oracle
        import synth
        self.oracle, self.n = oracle, n
        g = synth.rng(seed)
        self.codes, self.scales = synth.index_key_bytes(g, n)
        self.main = np.concatenate([g.integers(0, 256, size=(n, 256), dtype=np.uint8),
                                    g.integers(0x30, 0x39, size=(n, 32), dtype=np.uint8)], axis=1)
        self.sum_codes, self.sum_scales = oracle.block_summary(self.codes, self.scales, n)
        self.swa = synth.swa_rows(g, WIN)
        self.qs = [(synth.index_queries(g), synth.head_weights(g), synth.main_queries(g))
                   for _ in range(n_query_sets)]

    def run(self, n_queries: int) -> tuple[float, float]:
        o, n = self.oracle, self.n
        e0 = (n - 1) // 8 * 8
        t0 = time.perf_counter()
        for i in range(n_queries):
            q_idx, wh, q = self.qs[i % len(self.qs)]
            sc, ss = o.block_summary(self.codes[e0:n], self.scales[e0:n], n - e0)
            self.sum_codes[e0 // 8], self.sum_scales[e0 // 8] = sc[0], ss[0]
            pool = o.hisa_blocks(q_idx, wh, self.sum_codes, self.sum_scales, n, M_BLK)
            o.decode_query(o.REINDEX, t=n - 1, m=1, n_entries=n, main_kv=self.main, idx_codes=self.codes,
                           idx_scales=self.scales, q=q, swa=self.swa, swa_base=n - WIN, scale=1 / math.sqrt(D),
                           M=M_BLK, K=K_SEL, q_idx=q_idx, w_head=wh, pool_blocks=pool)
        dt = time.perf_counter() - t0
        return n_queries / dt, dt


class OracleLayer:
    """Oracle on the per-query work of a Full-mode layer over n entries of ratio
    m (index scan of every visible entry, top-2048 blocks, top-512, attention),
    optionally followed by Reuse layers on its selection and by Reindex groups
    (Reindex over its blocks + 3 Reuse).  Stored bytes drawn at random as in
    OracleHisa; each query's 128 window rows are one fixed set of rows."""

    def __init__(self, n: int, m: int, seed: int = 13, n_query_sets: int = 4):
        import numpy as np
        import oracle
        import synth
        self.oracle, self.n, self.m = oracle, n, m
        g = synth.rng(seed)
        self.codes, self.scales = synth.index_key_bytes(g, n)
        self.main = np.concatenate([g.integers(0, 256, size=(n, 256), dtype=np.uint8),
                                    g.integers(0x30, 0x39, size=(n, 32), dtype=np.uint8)], axis=1)
        self.swa = synth.swa_rows(g, WIN)
        self.qs = [(synth.index_queries(g), synth.head_weights(g), synth.main_queries(g))
                   for _ in range(n_query_sets)]

    def run(self, positions, reuse: int = 0, reindex_groups: int = 0) -> float:
        """Seconds for one query at each raw position in `positions`."""
        o = self.oracle
        common = dict(m=self.m, n_entries=self.n, main_kv=self.main, idx_codes=self.codes, idx_scales=self.scales,
                      swa=self.swa, scale=1 / math.sqrt(D), M=M_BLK, K=K_SEL)
        t0 = time.perf_counter()
        for i, t in enumerate(positions):
            q_idx, wh, q = self.qs[i % len(self.qs)]
            c = dict(common, t=int(t), swa_base=int(t) - (WIN - 1), q=q)
            pool, sel, _ = o.decode_query(o.FULL, q_idx=q_idx, w_head=wh, **c)
            for _ in range(reuse):
                o.decode_query(o.REUSE, sel=sel, **c)
            for _ in range(reindex_groups):
                _, sel2, _ = o.decode_query(o.REINDEX, q_idx=q_idx, w_head=wh, pool_blocks=pool, **c)
                for _ in range(3):
                    o.decode_query(o.REUSE, sel=sel2, **c)
        return time.perf_counter() - t0


def _oracle_line(value: float, unit: str, sample: str) -> dict:
    return {"value": value, "unit": unit, "cores": oracle_threads(), "kind": "oracle", "sample": sample}


def _decoder_oracle(args, N: int):
    """One token through the whole decoder chain: Full + 3 Reuse, 4 x (Reindex + 3 Reuse)."""
    if args.cpu_sample_queries <= 0:
        return None
    n_tok = max(1, args.cpu_sample_queries // 192)
    dt = OracleLayer(N, 1).run([N - 1] * n_tok, reuse=3, reindex_groups=4)
    return _oracle_line(20 * n_tok / dt, "query-token-layers/s",
                        f"{n_tok} query tokens x 20 layer calls over {N:,} entries (m=1) on a cache of random "
                        f"stored bytes, {dt:.1f} s")


def _prefill_oracle(args, P: int, T: int, N: int, m: int, reuse: int):
    """Evenly spaced queries of the chunk, each a Full query (+ `reuse` Reuse layers)."""
    if args.cpu_sample_queries <= 0:
        return None
    import numpy as np
    n_q = max(2, args.cpu_sample_queries // 24)
    pos = np.linspace(P, T - 1, n_q).round().astype(np.int64)
    dt = OracleLayer(N, m).run(pos, reuse=reuse)
    unit = "query-token-layers/s" if reuse else "query-tokens/s"
    return _oracle_line((1 + reuse) * n_q / dt, unit,
                        f"{n_q} evenly spaced queries of t = {P:,}..{T - 1:,} over {N:,} entries (m={m}), "
                        f"{1 + reuse} layer call(s) each, cache of random stored bytes, {dt:.1f} s")


def _cachewrite_oracle(args):
    """The oracle's cache write (C, the pinned binary32 order) on a sample of
    tokens of each of the 4 source layers."""
    if args.cpu_sample_queries <= 0:
        return None
    import oracle
    import synth
    n_tok = max(2, args.cpu_sample_queries * 64)
    g = synth.rng(17)
    w0, w1 = synth.compressor_weights(g)
    W = synth.index_projection(g)
    xs = [(synth.latents(g, n_tok), m) for m in (2, 2, 2, 1)]
    cs = oracle.rope_table(n_tok)
    t0 = time.perf_counter()
    for x, m in xs:
        oracle.compress_quantize(x, m, w0, w1, W, 0, cs=cs)
    dt = time.perf_counter() - t0
    return _oracle_line(4 * n_tok / dt, "tokens/s",
                        f"{n_tok:,} tokens of each of the 4 source layers (3 at m=2, 1 at m=1), {dt:.1f} s")


def oracle_threads() -> int:
    try:
        import numpy as np
        cfg = np.show_config(mode="dicts")
        _ = cfg
    except Exception:
        pass
    return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


def run_reference(args):
    rank, world, _ = dist_info()
    if rank != 0:
        return None
    per_step = 8
    chain = OracleChain()
    for _ in range(max(args.warmup, 0)):
        chain.run(1)
    dt = 0.0
    for _ in range(args.steps):
        dt += chain.run(per_step)[1]
    v = per_step * 4 * args.steps / dt
    sample = f"{per_step} query tokens per step: Reindex over a 16,384-entry pool + 3 Reuse attentions (oracle)"
    return {"metric": METRIC, "value": v, "unit": UNIT, "impl": "reference", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": "decode Reindex + 3 Reuse, 1,048,576 entries/seq, "
                                                        "batch 16 per layer call"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode1m",
                    choices=["decode1m", "full131k", "prefill8k", "cachewrite", "decoder1m", "prefillblock",
                             "hisa131k", "hisa1m"])
    ap.add_argument("--seq-len", type=int, default=1 << 20)
    ap.add_argument("--pipeline-distance", type=int, default=3)
    ap.add_argument("--cpu-sample-queries", type=int, default=768)
    ap.add_argument("--packed-selection", type=int, default=1,
                    help="decode: the Reindex call packs its selected entries for the Reuse calls (1) or not (0)")
    ap.add_argument("--lanes", type=int, default=10,
                    help="decode: stream + workspace lanes per layer slot")
    ap.add_argument("--swa-format", default="bf16", choices=["bf16", "fp8"],
                    help="decode: window rows as bf16 (the configuration) or E4M3 (the pages' FP8 window); "
                         "fp8 reports no end-to-end figure")
    ap.add_argument("--graph-cycles", type=int, default=0,
                    help="decode: pipeline cycles (of 3 d + 1 steps) per replayed CUDA graph; 0 = as many "
                         "as a timed window of --steps holds (at most 10)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup

    rank, world, local = dist_info()
    if args.impl == "reference":
        res = run_reference(args)
        if res is not None:
            print(json.dumps(res), flush=True)
        return

    import torch
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    import fp4_kv_cache_csa2_gb300 as csa2
    csa2.load()
    if args.workload != "decode1m":
        fn = {"full131k": run_full131k, "prefill8k": run_prefill8k, "cachewrite": run_cachewrite,
              "decoder1m": run_decoder1m, "prefillblock": run_prefillblock, "hisa131k": run_hisa131k,
              "hisa1m": run_hisa1m}[args.workload]
        line = fn(args, torch, csa2)
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    res = run_decode1m(args, torch, csa2)
    if rank == 0:
        line = {"metric": METRIC, "value": res.pop("value"), "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": res.pop("ms_per_step"), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": res.pop("dtype"), "data": "synthetic"}
        line.update(res)
        line["cpu_baseline"] = None
        if args.cpu_sample_queries > 0:
            cpu_v, cpu_dt = OracleChain(swa_fp8=args.swa_format == "fp8").run(args.cpu_sample_queries)
            line["cpu_baseline"] = {"value": cpu_v, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
                                    "sample": f"{args.cpu_sample_queries} query tokens x (Reindex over a 16,384-"
                                              f"entry pool + 3 Reuse attentions), {cpu_dt:.1f} s"}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
