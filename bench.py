#!/usr/bin/env python3
"""Benchmark: FP8 paged decode attention, tokens/s and HBM GB/s.

Workload (default): the concurrency-sweep point with 64 requests -- each
request has an 8192-token prompt already quantised into an e4m3 paged cache
(GQA 32 query / 8 KV heads, head_dim 128, page 16, pool sized for 64
requests x (8192 + 1000) tokens) -- decoding one token per request per step.
One step is the whole hot path on one batch:
    kvq_append_check, one launch of
        kvq_append (quantise the step's new K/V into the pages) and
        kvq_check_tags (batched page-tag integrity check -> abort mask)
    kvq_decode_attn (split paged attention, then the merge of split rows).
Step i appends generated token (offset + i) mod 1000 of every request, so
the context during the default run is ~8.6k-8.8k tokens, the mean context of
the 1000-token generation.  All inputs are seeded synthetic data drawn by
fp8_paged_kv_attn_gb300.inputs.  The KV cache read per step (~1.1 GB) is
larger than L2, so no explicit flush is needed between steps.

--impl reference times the CPU oracle (fp64, all host cores) on a bounded
sample of the same workload: each step is one request's decode step.

Prints ONE JSON line (rank 0).  Multi-GPU (torchrun): every rank runs its own
independent replica of the workload (requests are independent; no
collective on the data path); value = all ranks' tokens / max rank time.
"""
import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP8 paged decode attention: tokens/s and HBM GB/s (% of GB300 peak)"
DECODE_KERNEL_SOURCES = ["fp8_paged_kv_attn_gb300/csrc/decode_attn.cu",
                         "fp8_paged_kv_attn_gb300/csrc/decode_attn_mma.cuh",
                         "fp8_paged_kv_attn_gb300/csrc/decode_common.cuh",
                         "fp8_paged_kv_attn_gb300/csrc/kvq_device.cuh"]
TRAFFIC_PROFILE = "profiles/decode_attn_sweep_b64.json"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["kvq", "reference"], default="kvq")
    ap.add_argument("--batch", type=int, default=64)
    ap.add_argument("--kv", choices=["e4m3", "bf16"], default="e4m3")
    ap.add_argument("--check", choices=["on", "off"], default="on")
    ap.add_argument("--offset", type=int, default=400, help="first generated-token index")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--eager", action="store_true",
                    help="call the library per operation instead of replaying a CUDA graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--seed", type=int, default=2)
    ap.add_argument("--workload", choices=["ragged", "integrity", "8x8192", "prefill", "handoff",
                                           "pages", "wq"],
                    default=None,
                    help="time one of the other decode workloads (pools filled with random "
                         "finite e4m3 codes on the GPU; one JSON line, not the headline)")
    ap.add_argument("--wq-kind", choices=["stack", "large", "all"], default="all",
                    help="--workload wq: which weight set to time")
    ap.add_argument("--wq-m", type=int, default=0,
                    help="--workload wq: one token count instead of 1, 8, 16, 32, 64")
    ap.add_argument("--wq-w", choices=["int4", "e4m3", "both"], default="both",
                    help="--workload wq: which weight format")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip timing the 8x8192, integrity and ragged workloads in the "
                         "default run")
    ap.add_argument("--config-steps", type=int, default=50,
                    help="timed steps of each of those workloads in the default run")
    ap.add_argument("--config-warmup", type=int, default=5)
    ap.add_argument("--sustain-s", type=float, default=1.0,
                    help="seconds of back-to-back graph steps after the timed region (clock "
                         "record under steady load); 0 turns it off")
    ap.add_argument("--clocks-csv", default=None,
                    help="keep the raw nvidia-smi clock samples in this file")
    ap.add_argument("--no-parity-check", action="store_true",
                    help="skip comparing sampled rows of the last timed step with the oracle")
    ap.add_argument("--sweep-tokens", type=int, default=1000,
                    help="--sweep: generated tokens timed per point (all 1000 by default)")
    ap.add_argument("--sweep", action="store_true",
                    help="concurrency sweep 1/8/16/32/64 requests, e4m3 and bf16 KV at equal pool "
                         "bytes; one JSON line per point (not the headline line)")
    return ap.parse_args()


# ----------------------------------------------------------------------------
# distributed plumbing (barrier + max of times only)
# ----------------------------------------------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)
        return dist, rank, world, local
    return None, rank, world, local


def dist_max(dist, x: float) -> float:
    if dist is None:
        return x
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(dist):
    if dist is not None:
        dist.barrier()


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples of SM clock, utilisation, power and throttle
    reasons while the GPU measurements run.  The samples go to a temporary
    file (or `path`); the summary counts a sample as under load when the GPU
    reported at least 50% utilisation."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20, path=None):
        """Starts sampling every period_ms and returns once the sampler has
        written its first line, so that the measurements that follow are
        covered; samples written before that point are not counted."""
        self.proc = None
        self.skip = 0
        self.keep = path is not None
        if path is None:
            fd, path = tempfile.mkstemp(prefix=f"kvq_clocks_{gpu_index}_", suffix=".csv")
            os.close(fd)
        self.path = path
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(period_ms)],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        t0 = time.time()
        while time.time() - t0 < 5.0 and self.proc.poll() is None:
            with open(self.path) as f:
                n = sum(1 for _ in f)
            if n > 0:
                self.skip = n
                break
            time.sleep(0.01)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            lines = f.readlines()
        if not self.keep:
            os.unlink(self.path)
        for i, line in enumerate(lines):
            if i < self.skip:  # written before the measurements began
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                util = float(parts[4])
                rows.append((float(parts[1]), float(parts[2]), util, float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return None
        loaded = [r for r in rows if r[2] >= 50.0]
        use = loaded if loaded else rows
        reasons = sorted({self.REASONS[i] for r in use for i, v in enumerate(r[4])
                          if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in use),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": max(r[3] for r in use)}


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------

def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def code_only(text: str) -> str:
    """C++ source without its comments and with runs of whitespace collapsed,
    so that a comment-only edit keeps the hash (the kernel sources hold no
    string literal with // or /* in it)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def decode_source_sha() -> str:
    """Hash of the decode-attention kernel sources (code only), which the
    committed ncu traffic figure is tied to."""
    h = hashlib.sha256()
    for p in DECODE_KERNEL_SOURCES:
        with open(os.path.join(ROOT, p)) as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per decode-attention call from the committed ncu figure,
    only if it was taken on the current kernel source."""
    try:
        with open(os.path.join(ROOT, TRAFFIC_PROFILE)) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256_16") != decode_source_sha():
        return None
    return float(rec["traffic_bytes_per_call"])


def attn_kernels(B, D):
    """Kernels one kvq_decode_attn call launches for 8 kv heads a request:
    the split and combine kernels when the split kernel schedules the batch
    itself (head_dim 128, up to 4,608 requests), plus the plan kernel
    otherwise."""
    return 2 if D == 128 and B <= 4608 else 3


def attn_bytes(lens, Hq, Hkv, D, P, es):
    """Algorithmic bytes of one decode-attention call: every cached K and V
    element once, q in, out (fp32), and the block-table entries read."""
    lens = np.asarray(lens, dtype=np.int64)
    return int((lens * Hkv * D * 2 * es).sum() + len(lens) * Hq * D * (2 + 4)
               + ((lens + P - 1) // P * 4).sum())


# ----------------------------------------------------------------------------
# the decode step: packed inputs, eager calls or a replayed CUDA graph
# ----------------------------------------------------------------------------

class StepInputs:
    """The inputs of one decode step (q, k_new, v_new, pos, seq_lens) packed
    into one byte row, every field 256-byte aligned, so that a step's inputs
    are staged with a single copy (device to device, or host to device)."""

    def __init__(self, torch, B, Hq, Hkv, D):
        self.torch = torch
        spec = [("q", torch.bfloat16, (B, Hq, D), 2), ("k", torch.bfloat16, (B, Hkv, D), 2),
                ("v", torch.bfloat16, (B, Hkv, D), 2), ("pos", torch.int32, (B,), 4),
                ("lens", torch.int32, (B,), 4)]
        self.fields, off = [], 0
        for name, dt, shape, es in spec:
            n = int(np.prod(shape)) * es
            self.fields.append((name, off, n, dt, shape))
            off += -(-n // 256) * 256
        self.nbytes = off

    def views(self, row):
        return {name: row[o:o + n].view(dt).view(shape) for name, o, n, dt, shape in self.fields}

    def pack(self, steps):
        """steps: per step a dict field -> numpy array (bf16 fields as 16-bit
        bit patterns).  Returns a uint8 host tensor [len(steps), nbytes]."""
        torch = self.torch
        host = torch.zeros((len(steps), self.nbytes), dtype=torch.uint8)
        for i, st in enumerate(steps):
            for name, o, n, _, _ in self.fields:
                raw = np.ascontiguousarray(st[name]).view(np.uint8).reshape(-1)
                assert raw.size == n, (name, raw.size, n)
                host[i, o:o + n] = torch.from_numpy(raw)
        return host


class DecodeStep:
    """One decode step over a packed input row: kvq_append and
    kvq_check_tags in one launch (kvq_append_check, when `check`; the check
    writes `mask`; kvq_append alone otherwise) and kvq_decode_attn (which
    skips the requests `mask` flags, when a mask is given), through the
    library's Python binding.

    graph=True captures the step once over static buffers into a CUDA graph
    (the kernels are chained as programmatic dependents, which the
    capture keeps as programmatic edges); each step then stages its inputs
    with one copy into the static row and replays the graph.  A second graph
    holds the attention call alone, for timing it by itself.  graph=False
    calls the library eagerly on the step's own row."""

    def __init__(self, torch, kvq, cache, bt, P, sm_scale, packer, out, ws, err=None,
                 check=False, tags=None, exp_tags=None, mask=None, graph=True):
        self.torch, self.kvq, self.cache, self.bt, self.P = torch, kvq, cache, bt, P
        self.sm_scale, self.packer, self.out, self.ws, self.err = sm_scale, packer, out, ws, err
        self.check, self.tags, self.exp_tags, self.mask = check, tags, exp_tags, mask
        self.graph = graph
        B = bt.shape[0]
        self.req_idx = torch.arange(B, dtype=torch.int32, device="cuda")
        self.row = torch.zeros(packer.nbytes, dtype=torch.uint8, device="cuda")
        self.static = packer.views(self.row)
        self.g_step = self.g_attn = None

    # -- the library calls
    def append_check(self, v):
        kvq = self.kvq
        if self.check:
            kvq.kvq_append_check(self.cache, v["k"], v["v"], self.req_idx, v["pos"], self.bt,
                                 v["lens"], self.tags, self.exp_tags, self.mask,
                                 err_word=self.err)
        else:
            kvq.kvq_append(self.cache, v["k"], v["v"], self.req_idx, v["pos"], self.bt,
                           err_word=self.err)

    def attn(self, v):
        self.kvq.kvq_decode_attn(self.cache, v["q"], self.bt, v["lens"], self.out, self.ws,
                                 abort_mask=self.mask, sm_scale=self.sm_scale, err_word=self.err)

    def eager(self, v):
        self.append_check(v)
        self.attn(v)

    # -- graphs
    def capture(self, warm_row):
        """Runs the step eagerly on `warm_row` (fills the library's per-device
        caches), then captures both graphs on the static row."""
        torch = self.torch
        self.row.copy_(warm_row)
        self.eager(self.static)
        torch.cuda.synchronize()
        self.g_step = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_step):
            self.eager(self.static)
        self.g_attn = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_attn):
            self.attn(self.static)
        torch.cuda.synchronize()

    def run(self, row):
        """One whole step on a device row (staged into the graph's buffers)."""
        if self.graph:
            self.row.copy_(row, non_blocking=True)
            self.g_step.replay()
        else:
            self.eager(self.packer.views(row))

    def run_staged(self, host_row):
        """One whole step whose inputs come from pinned host memory."""
        self.row.copy_(host_row, non_blocking=True)
        if self.graph:
            self.g_step.replay()
        else:
            self.eager(self.static)

    def capture_flush_pair(self, flush):
        """Two more graphs for timing the attention call as it runs inside a
        step graph: the L2 flush alone, and the flush followed by the call.
        Their difference is the call's device time without the launch latency
        of a graph (which a step graph pays once for all its kernels)."""
        torch = self.torch
        self.g_f = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_f):
            flush()
        self.g_fa = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_fa):
            flush()
            self.attn(self.static)
        torch.cuda.synchronize()

    def run_attn_diff(self, row, ev, stream):
        """Stages the step's inputs, then the flush graph and the flush +
        attention graph, each between two recorded events (ev: four events)."""
        self.row.copy_(row, non_blocking=True)
        ev[0].record(stream)
        self.g_f.replay()
        ev[1].record(stream)
        ev[2].record(stream)
        self.g_fa.replay()
        ev[3].record(stream)

    def run_attn_timed(self, row, ev, stream):
        """The step's attention call alone between two recorded events (for
        the graph, the step's inputs are staged before the first event)."""
        if self.graph:
            self.row.copy_(row, non_blocking=True)
            ev[0].record(stream)
            self.g_attn.replay()
        else:
            self.append_check(self.packer.views(row))
            ev[0].record(stream)
            self.attn(self.packer.views(row))
        ev[1].record(stream)


class L2Flush:
    """Writes a buffer twice the size of L2 before a timed step whose inputs
    would otherwise stay L2-resident from one step to the next."""

    def __init__(self, torch):
        self.l2 = int(torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size)
        self.buf = torch.empty(self.l2 // 2, dtype=torch.int32, device="cuda")  # 2 x L2 bytes

    def __call__(self):
        self.buf.fill_(1)

    @staticmethod
    def needed(torch, kv_bytes_per_step):
        l2 = int(torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size)
        return kv_bytes_per_step < 2 * l2


def time_steps(torch, step, d_rows, warmup, steps, flush=None):
    """Warm-up steps, then `steps` whole steps, then each step's attention
    call timed alone.  Returns (ms per step, [ms per attention call],
    [ms per attention call in its own graph] or None).
    Without `flush` the whole steps run back to back in one timed region and
    each attention call is timed in its own graph.  With it, L2 is flushed
    before every timed step and each step is timed by its own pair of
    events; the attention call is timed (graph mode) as the difference of a
    graph holding the flush and the call and one holding the flush alone, so
    that the graph's own launch latency cancels (the call as it runs inside a
    step graph), and also in its own graph after a flush (launch latency
    included)."""
    stream = torch.cuda.current_stream()
    for i in range(warmup):
        step.eager(step.packer.views(d_rows[i]))
    if step.graph:
        step.capture(d_rows[max(warmup - 1, 0)])
        step.run(d_rows[max(warmup - 1, 0)])
        if flush is not None:
            step.capture_flush_pair(flush)
    torch.cuda.synchronize()

    def pairs(k=2):
        return [tuple(torch.cuda.Event(enable_timing=True) for _ in range(k))
                for _ in range(steps)]

    ev, es = pairs(), pairs()
    if flush is None:
        es[0][0].record(stream)
        for j in range(steps):
            if step.graph:
                step.run(d_rows[warmup + j])
            else:  # the eager loop times each attention call inside the step
                step.run_attn_timed(d_rows[warmup + j], ev[j], stream)
        es[0][1].record(stream)
    else:
        for j in range(steps):
            flush()
            es[j][0].record(stream)
            if step.graph:
                step.run(d_rows[warmup + j])
            else:
                step.eager(step.packer.views(d_rows[warmup + j]))
            es[j][1].record(stream)
    own = None
    if step.graph or flush is not None:
        for j in range(steps):
            if flush is not None:
                flush()
            step.run_attn_timed(d_rows[warmup + j], ev[j], stream)
    if step.graph and flush is not None:
        own = ev
        ev = pairs(4)
        for j in range(steps):
            step.run_attn_diff(d_rows[warmup + j], ev[j], stream)
    torch.cuda.synchronize()
    if flush is None:
        step_ms = es[0][0].elapsed_time(es[0][1]) / steps
    else:
        step_ms = statistics.mean(a.elapsed_time(b) for a, b in es)
    if own is None:
        return step_ms, [e[0].elapsed_time(e[1]) for e in ev], None
    return (step_ms, [e[2].elapsed_time(e[3]) - e[0].elapsed_time(e[1]) for e in ev],
            [e[0].elapsed_time(e[1]) for e in own])


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def run_gpu(args, dist, rank, world, local):
    import torch
    from fp8_paged_kv_attn_gb300 import inputs, kvq

    torch.cuda.set_device(local)
    kvq.load()
    kv_bytes = 1 if args.kv == "e4m3" else 2
    w = inputs.sweep(args.batch, kv_bytes=kv_bytes, seed=args.seed + rank)
    B, Hq, Hkv, D, P = w.B, w.Hq, w.Hkv, w.D, w.P
    steps_total = args.warmup + args.steps

    # --- cache: prompt K/V drawn on the host, quantised into pages on the GPU
    sources = w.kv_sources(threads=os.cpu_count() or 8)
    ks, vs = w.scales(sources)
    shape = w.pool_shape()
    pdt = torch.uint8 if kv_bytes == 1 else torch.bfloat16
    cache = kvq.KVCache(torch.zeros(shape, dtype=pdt, device="cuda"),
                        torch.zeros(shape, dtype=pdt, device="cuda"), float(ks), float(vs))
    bt = torch.from_numpy(w.block_table).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)

    for b, (k, v) in enumerate(sources):
        req, pos = w.context_tokens(b)
        kvq.kvq_append(cache, bf16(k).cuda(), bf16(v).cuda(), torch.from_numpy(req).cuda(),
                       torch.from_numpy(pos).cuda(), bt, err_word=err)
    torch.cuda.synchronize()
    kept_sources = {b: sources[b] for b in spot_check_requests(B)}
    del sources

    # --- per-step inputs, packed one row per step (device resident for the
    # kernel-time loop, pinned host memory for the end-to-end loop)
    gen = [(args.offset + i) % inputs.SWEEP_DECODE_STEPS for i in range(steps_total)]
    packer = StepInputs(torch, B, Hq, Hkv, D)
    host_len = []
    rows = []
    for gi in gen:
        q, k_new, v_new, _, pos = w.step_inputs(gi)
        host_len.append(w.seq_lens_after(gi))
        rows.append({"q": q, "k": k_new, "v": v_new, "pos": pos, "lens": host_len[-1]})
    h_rows = packer.pack(rows)
    d_rows = h_rows.cuda()
    del rows
    tags = torch.from_numpy(w.page_tags.view(np.int32)).cuda()
    exp_tags = torch.from_numpy(w.expected_tags.view(np.int32)).cuda()
    # the step's result, out (fp32) then the abort mask, in one buffer so that
    # the end-to-end loop reads it back with a single copy
    out_bytes = B * Hq * D * 4
    result_buf = torch.zeros(out_bytes + B, dtype=torch.uint8, device="cuda")
    out = result_buf[:out_bytes].view(torch.float32).view(B, Hq, D)
    mask = result_buf[out_bytes:]
    ws = kvq.workspace(B, Hq, Hkv, D)
    check = args.check == "on"
    graph = not args.eager
    stream = torch.cuda.current_stream()
    step = DecodeStep(torch, kvq, cache, bt, P, float(w.sm_scale), packer, out, ws, err=err,
                      check=check, tags=tags, exp_tags=exp_tags, mask=mask if check else None,
                      graph=graph)

    # the other decode workloads, set up before the measurements start (their
    # host-side set-up would otherwise leave the GPU idle inside them)
    extras = []
    if rank == 0 and world == 1 and not args.no_configs:
        for name in ("8x8192", "integrity", "ragged"):
            extras.append(WorkloadStep(torch, kvq, name, args.seed,
                                       args.config_warmup + args.config_steps,
                                       eager=args.eager))
        extras.append(HandoffStep(torch, kvq, args.seed))
        extras.append(WqStep(torch, kvq, args.seed))
        torch.cuda.synchronize()

    for i in range(args.warmup):
        step.eager(packer.views(d_rows[i]))
    if graph:
        last = d_rows[max(args.warmup - 1, 0)]
        step.capture(last)
        step.run(last)  # first replay (graph upload) outside the timed region
    torch.cuda.synchronize()

    def pairs(n=args.steps):
        return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(n)]

    # a step's KV smaller than 2 x L2 would stay cached from step to step:
    # then L2 is flushed before every timed step and each step is timed alone
    kv_step = attn_bytes(host_len[args.warmup], Hq, Hkv, D, P, kv_bytes)
    flush = L2Flush(torch) if L2Flush.needed(torch, kv_step) else None
    attn_ev, step_ev = pairs(), pairs()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    dist_barrier(dist)
    torch.cuda.synchronize()
    # clocks are sampled over every GPU measurement below: the timed steps,
    # the attention replays, the end-to-end loop, the sustained loop and the
    # other workloads
    clocks = ClockSampler(local, path=args.clocks_csv)
    torch.cuda.nvtx.range_push("timed")
    t_start.record(stream)
    for j in range(args.steps):
        if flush is not None:
            flush()
            step_ev[j][0].record(stream)
        if graph:
            step.run(d_rows[args.warmup + j])
        else:  # the eager loop times each attention call inside the step
            step.run_attn_timed(d_rows[args.warmup + j], attn_ev[j], stream)
        if flush is not None:
            step_ev[j][1].record(stream)
    t_end.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    if graph:
        # the attention graph alone over the same steps' inputs (every token
        # it reads was appended by the timed steps), events around each replay
        torch.cuda.nvtx.range_push("attn")
        for j in range(args.steps):
            if flush is not None:
                flush()
            step.run_attn_timed(d_rows[args.warmup + j], attn_ev[j], stream)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
    # the last timed step's output and abort mask, kept for the oracle check
    last_result = result_buf.clone()
    dist_barrier(dist)
    if flush is None:
        elapsed_ms = t_start.elapsed_time(t_end)
    else:
        elapsed_ms = sum(a.elapsed_time(b) for a, b in step_ev)
    elapsed_ms = dist_max(dist, elapsed_ms)
    attn_ms = [a.elapsed_time(b) for a, b in attn_ev]
    if int(err.item()) != 0:
        raise RuntimeError(f"device error bits {int(err.item()):#x}")
    if check and int(mask.sum().item()) != 0:
        raise RuntimeError("integrity check aborted requests on a clean workload")

    bytes_per_call = [attn_bytes(host_len[args.warmup + j], Hq, Hkv, D, P, kv_bytes)
                      for j in range(args.steps)]
    achieved = sum(bytes_per_call) / (sum(attn_ms) * 1e-3) / 1e9
    peak, peak_kind = measured_hbm_peak()

    # --- end to end: the step's inputs copied from pinned host memory, the
    # result (out + abort mask) read back, inside the timed region
    e2e = None
    if not args.no_e2e:
        h_pinned = h_rows.pin_memory()
        h2d = packer.nbytes
        d2h = result_buf.numel()

        def serial_e2e():
            """Copy in, step, copy out, one after another on one stream."""
            h_result = torch.empty(d2h, dtype=torch.uint8).pin_memory()
            torch.cuda.synchronize()
            dist_barrier(dist)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e2e_ev = pairs()
            e0.record(stream)
            for j in range(args.steps):
                if flush is not None:
                    flush()
                    e2e_ev[j][0].record(stream)
                step.run_staged(h_pinned[args.warmup + j])
                h_result.copy_(result_buf, non_blocking=True)
                if flush is not None:
                    e2e_ev[j][1].record(stream)
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) if flush is None else \
                sum(a.elapsed_time(b) for a, b in e2e_ev)
            return dist_max(dist, ms)

        def pipelined_e2e():
            """Two step graphs over two staging rows and result buffers (the
            cache, tables, tags and workspace are shared; the steps run in
            order on the compute stream).  Step j's input copy runs on one
            copy stream and its result copy on another, so they overlap the
            kernels of steps j - 1 and j + 1; each copy waits for the step
            that last used its buffer."""
            result2 = torch.zeros_like(result_buf)
            out2 = result2[:out_bytes].view(torch.float32).view(B, Hq, D)
            step2 = DecodeStep(torch, kvq, cache, bt, P, float(w.sm_scale), packer, out2, ws,
                               err=err, check=check, tags=tags, exp_tags=exp_tags,
                               mask=result2[out_bytes:] if check else None, graph=True)
            step2.capture(d_rows[max(args.warmup - 1, 0)])
            steps2, results = (step, step2), (result_buf, result2)
            h_res = [torch.empty(d2h, dtype=torch.uint8).pin_memory() for _ in range(2)]
            s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

            def ev():
                return torch.cuda.Event(enable_timing=False)
            ev_in, ev_done, ev_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]
            for b in range(2):
                ev_done[b].record(stream)
                ev_out[b].record(stream)
            torch.cuda.synchronize()
            dist_barrier(dist)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            s_in.wait_event(e0)
            for j in range(args.steps):
                b = j % 2
                with torch.cuda.stream(s_in):
                    s_in.wait_event(ev_done[b])  # the step that last read row b is done
                    steps2[b].row.copy_(h_pinned[args.warmup + j], non_blocking=True)
                    ev_in[b].record(s_in)
                stream.wait_event(ev_in[b])
                stream.wait_event(ev_out[b])  # result b of step j - 2 has been read back
                steps2[b].g_step.replay()
                ev_done[b].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_done[b])
                    h_res[b].copy_(results[b], non_blocking=True)
                    ev_out[b].record(s_out)
            stream.wait_event(ev_out[0])
            stream.wait_event(ev_out[1])
            e1.record(stream)
            torch.cuda.synchronize()
            # the last step's result as read back equals the device buffer
            last = (args.steps - 1) % 2
            if not torch.equal(h_res[last], results[last].cpu()):
                raise RuntimeError("pipelined end-to-end loop: result read back differs")
            return dist_max(dist, e0.elapsed_time(e1))

        # value: the serial loop, as an autoregressive decode runs (the next
        # step's inputs depend on this step's result).  pipelined_value: the
        # same copies overlapped with neighbouring steps, as a server with
        # independent work in flight could run them.
        e2e_ms = serial_e2e()
        e2e = {"value": round(world * B * args.steps / (e2e_ms * 1e-3), 1), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "mode": "serial: copy in, step, copy out on one stream"}
        if graph and flush is None:
            p_ms = pipelined_e2e()
            e2e["pipelined_value"] = round(world * B * args.steps / (p_ms * 1e-3), 1)
            e2e["pipelined_mode"] = ("each step's input copy (pinned host to device) and "
                                     "result copy (device to pinned host) on two copy streams, "
                                     "double-buffered, overlapping the neighbouring steps' "
                                     "kernels; all inside the timed region")

    # --- sustained: the same steps replayed back to back for about
    # args.sustain_s seconds (cycling over the timed steps' inputs), so that
    # the clock record covers a steady load, not only the short timed region
    sustained = None
    if args.sustain_s > 0 and graph:
        n = max(1, int(math.ceil(args.sustain_s / (elapsed_ms * 1e-3 / args.steps))))
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s0.record(stream)
        for j in range(n):
            if flush is not None:
                flush()
            step.run(d_rows[args.warmup + j % args.steps])
        s1.record(stream)
        torch.cuda.synchronize()
        sms = s0.elapsed_time(s1)
        sustained = {"steps": n, "ms": round(sms, 2), "ms_per_step": round(sms / n, 5),
                     "tokens_per_s": round(B * n / (sms * 1e-3), 1),
                     "l2": "flushed before every step (flush time included)"
                           if flush is not None else "no flush"}
        if int(err.item()) != 0:
            raise RuntimeError(f"device error bits {int(err.item()):#x}")

    # --- the other decode workloads, each timed in this process
    configs = {}
    for x in extras:
        rec = x.time(args.config_warmup, args.config_steps)
        configs[getattr(x, "name", "prefill_handoff")] = rec
    clk = clocks.stop()
    del extras

    value = world * B * args.steps / (elapsed_ms * 1e-3)
    ctx_mean = float(np.mean([host_len[args.warmup + j].mean() for j in range(args.steps)]))
    result = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(elapsed_ms / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded N(0,1) bf16 K/V with 1% outliers x20, quantised to e4m3 "
                "in the GPU's append kernel)",
        "config": {
            "workload": f"concurrency sweep point: {B} requests x 8192-token prompt + decode "
                        f"(generated tokens {gen[args.warmup]}..{gen[-1]}), GQA {Hq}/{Hkv}, "
                        f"head_dim {D}, page {P}, {args.kv} KV, integrity check {args.check}",
            "batch": B, "mean_context": round(ctx_mean, 1), "kv_dtype": args.kv,
            "pool_pages": w.num_pages, "page_size": P, "check": args.check,
            "l2": (f"inputs larger than L2 ({kv_step / 1e9:.2f} GB of KV read per step); no flush"
                   if flush is None else
                   f"L2 ({flush.l2 >> 20} MB) flushed before every timed step and attention "
                   f"call ({kv_step / 1e6:.0f} MB of KV per step); each timed by its own events"),
            "step": ("kvq_append_check (append + tag check, one launch) + kvq_decode_attn"
                     if check else "kvq_append + kvq_decode_attn"),
            "launch": "CUDA graph per step (inputs staged with one device copy; the step's "
                      "kernels chained as programmatic dependents)" if graph
                      else "eager library calls",
        },
        "roofline": {
            "bound": "hbm",
            "kernel": "kvq_decode_attn (split + combine; + plan above 4,608 requests), CUDA events around each call"
                      + (" (its own graph, replayed per step)" if graph else ""),
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
            else "fallback 6.8 TB/s",
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": profiled_traffic(),
            "bytes_per_call": int(statistics.mean(bytes_per_call)),
            "ms_per_call": round(statistics.mean(attn_ms), 5),
            "ms_per_call_median": round(statistics.median(attn_ms), 5),
            "ms_per_call_p95": round(float(np.percentile(attn_ms, 95)), 5),
        },
        "gpu_launches": args.steps * (1 + (1 if check else 0) + attn_kernels(B, D)),
        "clocks": clk,
    }
    if e2e is not None:
        result["e2e"] = e2e
    if sustained is not None:
        result["sustained"] = sustained
    if configs:
        result["configs"] = configs
    if rank == 0 and not args.no_parity_check:
        result["parity_check"] = oracle_spot_check(
            args, w, ks, vs, kv_bytes, kept_sources, packer, h_rows, gen, host_len,
            last_result[:out_bytes].view(torch.float32).view(B, Hq, D).cpu().numpy(),
            last_result[out_bytes:].cpu().numpy())
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args, w, ks, vs, args.cpu_seconds)
    return result


# ----------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ----------------------------------------------------------------------------

class OracleRequestStep:
    """One request's decode step on the CPU oracle: append its new token,
    check its page tags, attend for every query head."""

    def __init__(self, w, b, ks, vs):
        import oracle
        self.oracle = oracle
        self.w, self.b, self.ks, self.vs = w, b, ks, vs
        shape = w.pool_shape()
        self.kp = np.zeros(shape, dtype=np.uint8)
        self.vp = np.zeros(shape, dtype=np.uint8)
        k, v = w.kv_source(b)
        req, pos = w.context_tokens(b)
        oracle.quant_append(oracle.KV_E4M3, self.kp, self.vp, ks, vs, k, v, req, pos,
                            w.block_table)
        self.bt1 = w.block_table[b:b + 1]

    def run(self, gen_index, nthreads):
        o, w, b = self.oracle, self.w, self.b
        q, k_new, v_new, _, pos = w.step_inputs(gen_index)
        o.quant_append(o.KV_E4M3, self.kp, self.vp, self.ks, self.vs, k_new[b:b + 1],
                       v_new[b:b + 1], np.zeros(1, np.int32), pos[b:b + 1], self.bt1)
        lens = w.seq_lens_after(gen_index)[b:b + 1]
        mask = o.check_tags(self.bt1, lens, w.P, w.page_tags, w.expected_tags[b:b + 1])
        out, err = o.decode_attn(o.KV_E4M3, self.kp, self.vp, self.ks, self.vs, q[b:b + 1],
                                 self.bt1, lens, abort_mask=mask, sm_scale=w.sm_scale,
                                 nthreads=nthreads)
        return out


def spot_check_requests(B):
    """Requests whose output rows the default run checks against the oracle."""
    return sorted({0, B // 2, B - 1})


def _bf16_bits(t):
    return t.contiguous().view(__import__("torch").int16).numpy().view(np.uint16)


def oracle_spot_check(args, w, ks, vs, kv_bytes, sources, packer, h_rows, gen, host_len,
                      out_last, mask_last):
    """Every output row of a few requests after the last timed step, against
    the CPU oracle (fp64), and the whole abort mask, bit for bit.  The oracle's
    pools hold those requests' prompts and every token the run appended for
    them, in the run's order (warm-up steps, then the timed steps); the last
    step's q, lengths and tags give the expected rows.  A mismatch fails the
    run."""
    import oracle
    reqs = sorted(sources)
    sel = np.array(reqs, dtype=np.int32)
    dt = oracle.KV_E4M3 if kv_bytes == 1 else oracle.KV_BF16
    shape = w.pool_shape()
    hk = np.zeros(shape, dtype=np.uint8 if kv_bytes == 1 else np.uint16)
    hv = np.zeros_like(hk)
    for b in reqs:
        k, v = sources[b]
        req, pos = w.context_tokens(b)
        if oracle.quant_append(dt, hk, hv, ks, vs, k, v, req, pos, w.block_table) != 0:
            raise RuntimeError("oracle append of the prompt failed")
    n_run = args.warmup + args.steps
    for i in range(n_run):
        f = packer.views(h_rows[i])
        kb, vb = _bf16_bits(f["k"]), _bf16_bits(f["v"])
        pos = f["pos"].numpy()
        if oracle.quant_append(dt, hk, hv, ks, vs, np.ascontiguousarray(kb[sel]),
                               np.ascontiguousarray(vb[sel]), sel,
                               np.ascontiguousarray(pos[sel]), w.block_table) != 0:
            raise RuntimeError("oracle append of a step failed")
    last = packer.views(h_rows[n_run - 1])
    q = _bf16_bits(last["q"])
    lens = last["lens"].numpy().copy()
    check = args.check == "on"
    ref_mask = oracle.check_tags(w.block_table, lens, w.P, w.page_tags, w.expected_tags) \
        if check else np.zeros(w.B, dtype=np.uint8)
    mask_ok = (not check) or bool(np.array_equal(mask_last, ref_mask))
    rows = [(b, h) for b in reqs for h in range(w.Hq)]
    ref, oerr = oracle.decode_attn(dt, hk, hv, ks, vs, q, w.block_table, lens,
                                   abort_mask=ref_mask, sm_scale=w.sm_scale, rows=rows,
                                   nthreads=oracle_threads())
    got = out_last[sel].astype(np.float64)
    exp = ref[sel].astype(np.float64)
    err = np.abs(got - exp)
    tol = 1e-3 + 1e-3 * np.abs(exp)
    worst = float(np.max(err / tol))
    res = {"requests": reqs, "rows": len(rows), "step_generated_token": int(gen[n_run - 1]),
           "context": [int(lens[b]) for b in reqs], "max_abs_err": float(err.max()),
           "max_err_over_tol": round(worst, 5), "tol": "1e-3 + 1e-3*|ref| (fp64 oracle)",
           "abort_mask_bit_exact": mask_ok, "ok": bool(worst <= 1.0 and mask_ok and oerr == 0)}
    if not res["ok"]:
        raise RuntimeError(f"the last timed step differs from the oracle: {res}")
    return res


def oracle_threads():
    import oracle
    n = os.cpu_count() or 1
    return n if oracle.has_openmp() else 1


def cpu_baseline(args, w, ks, vs, seconds):
    nthreads = oracle_threads()
    done, t_total, b = 0, 0.0, 0
    gi = args.offset
    while t_total < seconds and b < w.B:
        st = OracleRequestStep(w, b, ks, vs)
        t0 = time.perf_counter()
        st.run(gi, nthreads)
        t_total += time.perf_counter() - t0
        done += 1
        b += 1
    return {"value": round(done / t_total, 3), "unit": "tokens/s", "cores": nthreads,
            "kind": "oracle",
            "sample": f"{done} requests' decode step (append + tag check + fp64 attention over "
                      f"~{int(w.ctx_lens[0]) + gi + 1} tokens, {w.Hq} heads), "
                      f"{t_total:.1f} s of CPU time"}


def run_reference(args, rank):
    from fp8_paged_kv_attn_gb300 import inputs
    w = inputs.sweep(args.batch, kv_bytes=1, seed=args.seed)
    # scales of the full workload need every request's prompt; the sample uses
    # request 0's own amax, which is what per-tensor calibration of that
    # request alone would give
    k0, v0 = w.kv_source(0)
    ks = inputs.scale_from_amax(inputs.amax_bf16(k0))
    vs = inputs.scale_from_amax(inputs.amax_bf16(v0))
    nthreads = oracle_threads()
    st = OracleRequestStep(w, 0, ks, vs)
    for i in range(args.warmup):
        st.run((args.offset + i) % inputs.SWEEP_DECODE_STEPS, nthreads)
    t0 = time.perf_counter()
    for j in range(args.steps):
        st.run((args.offset + args.warmup + j) % inputs.SWEEP_DECODE_STEPS, nthreads)
    dt = time.perf_counter() - t0
    value = args.steps / dt
    sample = (f"each step: one request's decode step (append + tag check + fp64 attention, "
              f"{w.Hq} heads, ~{8192 + args.offset} tokens) of the {args.batch}-request sweep")
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"concurrency sweep point ({args.batch} requests), one request "
                               f"per step on the CPU oracle", "batch": 1},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": nthreads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_sweep(args):
    """FP8 vs BF16 KV over 1..64 concurrent requests at equal pool bytes (the
    pages' decode table shape: 8192-token prompts, 1000 generated tokens).
    Each point runs the whole generation: `--sweep-tokens` (default all
    1000) decode steps (append + attention, no tag check), timed after
    `warmup` steps that append the first generated tokens (re-appended, same
    values, by the timed steps), and reports the mean over the generation."""
    import torch
    from fp8_paged_kv_attn_gb300 import inputs, kvq

    kvq.load()
    peak, _ = measured_hbm_peak()
    ref = inputs.sweep(64, kv_bytes=1, seed=args.seed)
    sources = ref.kv_sources(threads=os.cpu_count() or 8)
    ks, vs = ref.scales(sources)
    n_gen = min(args.sweep_tokens, inputs.SWEEP_DECODE_STEPS)

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)

    for kv in ("e4m3", "bf16"):
        kv_bytes = 1 if kv == "e4m3" else 2
        for B in (1, 8, 16, 32, 64):
            try:
                w = inputs.sweep(B, kv_bytes=kv_bytes, seed=args.seed)
            except MemoryError as e:
                print(json.dumps({"sweep": True, "kv": kv, "batch": B, "result": "OOM",
                                  "why": str(e)}), flush=True)
                continue
            shape = w.pool_shape()
            pdt = torch.uint8 if kv_bytes == 1 else torch.bfloat16
            cache = kvq.KVCache(torch.zeros(shape, dtype=pdt, device="cuda"),
                                torch.zeros(shape, dtype=pdt, device="cuda"), float(ks), float(vs))
            bt = torch.from_numpy(w.block_table).cuda()
            for b in range(B):
                k, v = sources[b]
                req, pos = w.context_tokens(b)
                kvq.kvq_append(cache, bf16(k).cuda(), bf16(v).cuda(), torch.from_numpy(req).cuda(),
                               torch.from_numpy(pos).cuda(), bt)
            # warm-up steps append generated tokens 0 .. W-1; the timed steps
            # then run the whole generation, tokens 0 .. n_gen-1
            gen = list(range(args.warmup)) + list(range(n_gen))
            packer = StepInputs(torch, B, w.Hq, w.Hkv, w.D)
            lens = [w.seq_lens_after(gi) for gi in gen]
            rows = []
            for gi, ln in zip(gen, lens):
                q, k_new, v_new, _, pos = w.step_inputs(gi)
                rows.append({"q": q, "k": k_new, "v": v_new, "pos": pos, "lens": ln})
            d_rows = packer.pack(rows).cuda()
            del rows
            out = torch.empty((B, w.Hq, w.D), dtype=torch.float32, device="cuda")
            ws = kvq.workspace(B, w.Hq, w.Hkv, w.D)
            step = DecodeStep(torch, kvq, cache, bt, w.P, float(w.sm_scale), packer, out, ws,
                              graph=not args.eager)
            byts = [attn_bytes(lens[i], w.Hq, w.Hkv, w.D, w.P, kv_bytes)
                    for i in range(args.warmup, len(gen))]
            flush = L2Flush(torch) if L2Flush.needed(torch, byts[0]) else None
            step_ms, attn_ms, attn_own = time_steps(torch, step, d_rows, args.warmup, n_gen,
                                                    flush)
            gbs = sum(byts) / (sum(attn_ms) * 1e-3) / 1e9
            line = {"sweep": True, "kv": kv, "batch": B, "generated_tokens": n_gen,
                    "tokens_per_s": round(B / (step_ms * 1e-3), 1),
                    "ms_per_step": round(step_ms, 5),
                    "attn_us": round(statistics.mean(attn_ms) * 1e3, 2),
                    "attn_us_p95": round(float(np.percentile(attn_ms, 95)) * 1e3, 2),
                    "attn_GBs": round(gbs, 1), "frac_of_measured_peak": round(gbs / peak, 4),
                    "l2": "flushed before each step" if flush else "KV larger than 2 x L2; no flush",
                    "attn_timing": ("difference of a graph of (L2 flush, call) and one of the "
                                    "flush alone" if attn_own else "the call's own graph"),
                    "pool_pages": w.num_pages,
                    "mean_context": round(float(np.mean([x.mean() for x in lens[args.warmup:]])), 1)}
            if attn_own:
                line["attn_us_own_graph"] = round(statistics.mean(attn_own) * 1e3, 2)
            if flush is not None:  # the same steps back to back, L2 warm, for comparison
                wstep, wattn, _ = time_steps(torch, step, d_rows, args.warmup, n_gen)
                line["tokens_per_s_warm"] = round(B / (wstep * 1e-3), 1)
                line["attn_us_warm"] = round(statistics.mean(wattn) * 1e3, 2)
            print(json.dumps(line), flush=True)
            del cache, d_rows


WORKLOADS = {"ragged": "ragged", "integrity": "integrity", "8x8192": "cfg8x8k"}


class WorkloadStep:
    """One of the other decode workloads (ragged: page 64, 8 query heads per
    kv head; integrity: 256 requests, stale tags, check -> mask -> attention;
    8x8192: one decode step of 8 requests x 8192 tokens) set up on the GPU
    for timing.  The cache holds random finite e4m3 codes written on the GPU
    (timing does not depend on the values; the parity tests cover these
    workloads with real data).  Every step stages the same inputs."""

    def __init__(self, torch, kvq, name, seed, rows_needed, eager=False):
        from fp8_paged_kv_attn_gb300 import inputs
        self.torch, self.kvq, self.name, self.eager = torch, kvq, name, eager
        w = getattr(inputs, WORKLOADS[name])()
        self.w = w
        B, Hq, Hkv, D, P = w.B, w.Hq, w.Hkv, w.D, w.P
        gen = torch.Generator(device="cuda").manual_seed(seed)
        pools = [torch.randint(0, 0x77, w.pool_shape(), dtype=torch.uint8, device="cuda",
                               generator=gen) for _ in range(2)]
        self.cache = kvq.KVCache(pools[0], pools[1], 0.01, 0.01)
        self.bt = torch.from_numpy(w.block_table).cuda()
        self.tags = torch.from_numpy(w.page_tags.view(np.int32)).cuda()
        self.exp_tags = torch.from_numpy(w.expected_tags.view(np.int32)).cuda()
        self.lens = w.seq_lens_after(0)
        q, k_new, v_new, req, pos = w.step_inputs(0)
        assert np.array_equal(req, np.arange(B, dtype=np.int32))
        self.packer = StepInputs(torch, B, Hq, Hkv, D)
        row = self.packer.pack([{"q": q, "k": k_new, "v": v_new, "pos": pos,
                                 "lens": self.lens}]).cuda()
        self.rows = row.expand(rows_needed, -1)  # the same step inputs every step
        self.mask = torch.zeros(B, dtype=torch.uint8, device="cuda")
        self.out = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
        self.ws = kvq.workspace(B, Hq, Hkv, D)
        self.flush = L2Flush(torch) if L2Flush.needed(
            torch, attn_bytes(self.lens, Hq, Hkv, D, P, 1)) else None

    def time(self, warmup, steps):
        """Times `steps` whole steps with the check, then the same without it
        but with the mask it produced (both arms attend the same requests, so
        the difference is the check alone).  Returns the result record."""
        torch, w = self.torch, self.w
        B, Hq, Hkv, D, P = w.B, w.Hq, w.Hkv, w.D, w.P

        def run(check):
            step = DecodeStep(torch, self.kvq, self.cache, self.bt, P, float(w.sm_scale),
                              self.packer, self.out, self.ws, check=check, tags=self.tags,
                              exp_tags=self.exp_tags, mask=self.mask, graph=not self.eager)
            step_ms, attn_ms, own = time_steps(torch, step, self.rows, warmup, steps, self.flush)
            return step_ms, statistics.mean(attn_ms), (statistics.mean(own) if own else None)

        step_on, attn_on, own_on = run(True)
        step_off, attn_off, _ = run(False)
        peak, _ = measured_hbm_peak()
        aborted = int(self.mask.sum().item())
        alive = (self.mask.cpu().numpy() == 0)
        byts = attn_bytes(self.lens[alive], Hq, Hkv, D, P, 1)
        gbs = byts / (attn_on * 1e-3) / 1e9
        res = {"workload": w.name, "batch": B, "tokens": int(self.lens.sum()), "Hq": Hq,
               "Hkv": Hkv, "page_size": P, "steps": steps,
               "tokens_per_s": round(B / (step_on * 1e-3), 1),
               "step_ms_with_check": round(step_on, 5),
               "attn_us_with_check": round(attn_on * 1e3, 2),
               "attn_GBs": round(gbs, 1), "frac_of_measured_peak": round(gbs / peak, 4),
               "aborted_requests": aborted,
               "l2": "flushed before each step" if self.flush else
                     "KV larger than 2 x L2; no flush",
               "attn_timing": ("difference of a graph of (L2 flush, call) and one of the flush "
                               "alone" if own_on else "the call's own graph")}
        if own_on:
            res["attn_us_own_graph"] = round(own_on * 1e3, 2)
            res["frac_own_graph"] = round(byts / (own_on * 1e-3) / 1e9 / peak, 4)
        if self.name == "integrity":
            res["step_ms_without_check"] = round(step_off, 5)
            res["check_overhead_pct_of_step"] = round(100 * (step_on - step_off) / step_off, 2)
        return res


def run_workload(args):
    """Decode-step timing on one of the other workloads (WorkloadStep), one
    JSON line."""
    import torch
    from fp8_paged_kv_attn_gb300 import kvq

    kvq.load()
    ws = WorkloadStep(torch, kvq, args.workload, args.seed, args.warmup + args.steps,
                      eager=args.eager)
    print(json.dumps(ws.time(args.warmup, args.steps)), flush=True)


def run_prefill(args):
    """The prefill -> decode handoff: the `--batch` (default 64) requests'
    whole 8192-token BF16 prompts (at 64: 524,288 tokens, 1.07 GB each of K
    and V) quantised into e4m3 pages by ONE kvq_append call, timed with CUDA
    events per call; then the same into a BF16 pool of as many pages (a
    paged copy), for comparison."""
    import torch
    from fp8_paged_kv_attn_gb300 import inputs, kvq

    kvq.load()
    peak, _ = measured_hbm_peak()
    w = inputs.sweep(args.batch, kv_bytes=1, seed=args.seed)
    sources = w.kv_sources(threads=os.cpu_count() or 8)
    ks, vs = w.scales(sources)

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()

    k_all = bf16(np.concatenate([k for k, _ in sources]))
    v_all = bf16(np.concatenate([v for _, v in sources]))
    toks = [w.context_tokens(b) for b in range(w.B)]
    req = torch.from_numpy(np.concatenate([t[0] for t in toks])).cuda()
    pos = torch.from_numpy(np.concatenate([t[1] for t in toks])).cuda()
    del sources, toks
    N = int(req.shape[0])
    bt = torch.from_numpy(w.block_table).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    for kv, es, pdt in (("e4m3", 1, torch.uint8), ("bf16", 2, torch.bfloat16)):
        shape = w.pool_shape()
        cache = kvq.KVCache(torch.zeros(shape, dtype=pdt, device="cuda"),
                            torch.zeros(shape, dtype=pdt, device="cuda"), float(ks), float(vs))
        for _ in range(args.warmup):
            kvq.kvq_append(cache, k_all, v_all, req, pos, bt, err_word=err)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        torch.cuda.synchronize()
        for e in ev:
            e[0].record(stream)
            kvq.kvq_append(cache, k_all, v_all, req, pos, bt, err_word=err)
            e[1].record(stream)
        torch.cuda.synchronize()
        if int(err.item()) != 0:
            raise RuntimeError(f"device error bits {int(err.item()):#x}")
        ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        # K and V read as bf16, written as codes; req_idx and pos read
        byts = N * w.Hkv * w.D * 2 * (2 + es) + N * 8
        print(json.dumps({"workload": f"prefill_handoff_{w.B}x8192", "kv": kv, "tokens": N,
                          "Hkv": w.Hkv, "D": w.D, "page_size": w.P, "steps": args.steps,
                          "us_per_call": round(ms * 1e3, 2),
                          "tokens_per_s": round(N / (ms * 1e-3), 1),
                          "GBs": round(byts / (ms * 1e-3) / 1e9, 1),
                          "frac_of_measured_peak": round(byts / (ms * 1e-3) / 1e9 / peak, 4),
                          "bytes_per_call": byts}), flush=True)
        del cache


class HandoffStep:
    """The prefill -> decode handoff of the sweep's 64 requests x 8192-token
    prompts in one kvq_handoff_pages call: a BF16 prefill pool of 64-token
    pages into the e4m3 decode pool of 64 requests x 575 pages of 16 tokens.
    The prefill pool holds seeded N(0,1) bf16 values with 1% outliers x20
    (the decode workloads' recipe, written on the GPU) and the e4m3 scales
    are amax / 448 of those values, so the codes and the quantiser's
    division fallback (elements near an e4m3 rounding boundary) behave as on
    real data; the parity tests cover the values."""

    def __init__(self, torch, kvq, seed, B=64):
        from fp8_paged_kv_attn_gb300 import inputs
        self.torch, self.kvq = torch, kvq
        h = inputs.handoff(seed=seed, B=B)
        self.h = h
        gen = torch.Generator(device="cuda").manual_seed(seed)

        def bf16_pool():
            z = torch.randn(h.src_shape(), device="cuda", generator=gen)
            out = torch.rand(h.src_shape(), device="cuda", generator=gen) < 0.01
            return (z * (1.0 + 19.0 * out)).to(torch.bfloat16)

        self.src = kvq.KVCache(bf16_pool(), bf16_pool())
        k_scale = float(self.src.k_pool.abs().max().float()) / 448.0
        v_scale = float(self.src.v_pool.abs().max().float()) / 448.0
        self.dst = kvq.KVCache(torch.zeros(h.dst_shape(), dtype=torch.uint8, device="cuda"),
                               torch.zeros(h.dst_shape(), dtype=torch.uint8, device="cuda"),
                               k_scale, v_scale)
        self.sbt = torch.from_numpy(h.src_block_table).cuda()
        self.dbt = torch.from_numpy(h.dst_block_table).cuda()
        self.count = torch.from_numpy(h.count).cuda()
        self.first = torch.from_numpy(h.first).cuda()
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.tokens = int(h.count.sum())
        # read bf16 K and V, write e4m3 codes; one block-table entry per page
        self.bytes = (self.tokens * h.Hkv * h.D * 2 * (2 + 1)
                      + int(sum(-(-int(c) // h.src_P) + -(-int(c) // h.dst_P) for c in h.count)) * 4)

    def call(self):
        self.kvq.kvq_handoff_pages(self.src, self.sbt, self.dst, self.dbt, self.count,
                                   first=self.first, err_word=self.err)

    def time(self, warmup, steps):
        torch = self.torch
        stream = torch.cuda.current_stream()
        for _ in range(warmup):
            self.call()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        torch.cuda.synchronize()
        for a, b in ev:
            a.record(stream)
            self.call()
            b.record(stream)
        torch.cuda.synchronize()
        if int(self.err.item()) != 0:
            raise RuntimeError(f"device error bits {int(self.err.item()):#x}")
        peak, _ = measured_hbm_peak()
        ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        gbs = self.bytes / (ms * 1e-3) / 1e9
        h = self.h
        return {"workload": f"prefill_handoff_{h.B}x8192_bf16p{h.src_P}_to_e4m3p{h.dst_P}",
                "tokens": self.tokens, "Hkv": h.Hkv, "D": h.D, "steps": steps,
                "us_per_call": round(ms * 1e3, 2), "tokens_per_s": round(self.tokens / (ms * 1e-3), 1),
                "GBs": round(gbs, 1), "frac_of_measured_peak": round(gbs / peak, 4),
                "bytes_per_call": self.bytes,
                "l2": "inputs larger than L2 (3.2 GB per call); no flush"}


def run_handoff(args):
    import torch
    from fp8_paged_kv_attn_gb300 import kvq
    kvq.load()
    print(json.dumps(HandoffStep(torch, kvq, args.seed, args.batch).time(args.warmup, args.steps)),
          flush=True)


def run_pages(args):
    """The page allocator (kvq_pages_update), one line per scenario: the
    batches of a decode step and of admission.  Each scenario is K calls
    captured in one CUDA graph; the allocator state is restored from a
    snapshot before every replay and only the replay is timed (CUDA events),
    so the per-call figure is device time, not the Python binding's."""
    import torch
    from fp8_paged_kv_attn_gb300 import kvq

    kvq.load()
    rng = np.random.default_rng(args.seed)
    stream = torch.cuda.current_stream()

    def state(num_pages, B, MP):
        return kvq.PageState(
            torch.from_numpy(rng.permutation(num_pages).astype(np.int32)).cuda(),
            torch.tensor([num_pages], dtype=torch.int32, device="cuda"),
            torch.zeros(num_pages, dtype=torch.int32, device="cuda"),
            torch.full((B, MP), -1, dtype=torch.int32, device="cuda"),
            torch.zeros((B, MP), dtype=torch.int32, device="cuda"))

    def i32(x):
        return torch.tensor(x, dtype=torch.int32, device="cuda")

    def timed(name, st, calls, pages_per_call, reps=20):
        """calls: list of kwargs for kvq_pages_update, run in order."""
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        snap = [t.clone() for t in (st.free_stack, st.free_count, st.page_tags, st.block_table,
                                    st.expected_tags)]

        def restore():
            for t, s0 in zip((st.free_stack, st.free_count, st.page_tags, st.block_table,
                              st.expected_tags), snap):
                t.copy_(s0)

        def run():
            for kw in calls:
                kvq.kvq_pages_update(st, err_word=err, **kw)

        run()  # eager warm-up (also checks the calls)
        torch.cuda.synchronize()
        bad = int(err.item()) & ~kvq.ERRBIT_EXHAUSTED
        if bad:
            raise RuntimeError(f"{name}: device error bits {bad:#x}")
        restore()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        for e in ev:
            restore()
            e[0].record(stream)
            g.replay()
            e[1].record(stream)
        torch.cuda.synchronize()
        us = statistics.median(a.elapsed_time(b) for a, b in ev) * 1e3 / len(calls)
        print(json.dumps({"workload": f"pages_{name}", "calls_per_graph": len(calls),
                          "us_per_call": round(us, 3), "pages_per_call": pages_per_call,
                          "pages_per_s": round(pages_per_call / (us * 1e-6), 1),
                          "reps": reps}), flush=True)

    # decode-step growth: 16 of 256 live requests cross into a new page
    st = state(65536, 256, 1024)
    live = rng.choice(256, 16, replace=False).astype(np.int32)
    calls = [dict(acq_req=i32(live), acq_first=i32(np.full(16, c, np.int32)),
                  acq_npages=i32(np.ones(16, np.int32)),
                  acq_ok=torch.zeros(16, dtype=torch.uint8, device="cuda")) for c in range(50)]
    timed("grow_16x1", st, calls, 16)

    # turnover: a finished 8k-token request (512 pages) leaves, a new one arrives
    st = state(65536, 256, 1024)
    setup_ok = torch.zeros(1, dtype=torch.uint8, device="cuda")
    kvq.kvq_pages_update(st, acq_req=i32([0]), acq_first=i32([0]), acq_npages=i32([512]),
                         acq_ok=setup_ok)
    calls = []
    for c in range(50):
        a, b = (0, 1) if c % 2 == 0 else (1, 0)
        calls.append(dict(rel_req=i32([a]), rel_npages=i32([512]), acq_req=i32([b]),
                          acq_first=i32([0]), acq_npages=i32([512]),
                          acq_ok=torch.zeros(1, dtype=torch.uint8, device="cuda")))
    timed("turnover_512", st, calls, 1024)

    # admission of 64 requests x 575 pages (the sweep pool), then its release
    st = state(36800, 64, 575)
    timed("admit_64x575", st, [dict(acq_req=i32(np.arange(64)), acq_first=i32(np.zeros(64)),
                                    acq_npages=i32(np.full(64, 575)),
                                    acq_ok=torch.zeros(64, dtype=torch.uint8, device="cuda"))],
          36800)
    st = state(36800, 64, 575)
    kvq.kvq_pages_update(st, acq_req=i32(np.arange(64)), acq_first=i32(np.zeros(64)),
                         acq_npages=i32(np.full(64, 575)),
                         acq_ok=torch.zeros(64, dtype=torch.uint8, device="cuda"))
    timed("release_64x575", st, [dict(rel_req=i32(np.arange(64)),
                                      rel_npages=i32(np.full(64, 575)))], 36800)


# GLM-like projection shapes at 8-way tensor parallelism (synthetic): hidden
# 5120, 96 query + 8 kv heads of 128, dense MLP 12288: (N, K) per layer
WQ_LAYER = [("qkv", 1792, 5120), ("o", 5120, 1536), ("gate_up", 3072, 5120), ("down", 5120, 1536)]
WQ_LAYERS = 40


def wq_weights(torch, kvq, gen, wdtype, N, K):
    """Seeded random quantised weights [N, K] and their scales; returns (w, scales, bytes)."""
    if wdtype == kvq.W_INT4:
        w = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device="cuda", generator=gen)
        s = torch.full((N, K // 128), 0x3C00, dtype=torch.int16, device="cuda")
        return w, s, N * K // 2 + N * (K // 128) * 2
    w = torch.randint(0, 0x77, (N, K), dtype=torch.uint8, device="cuda", generator=gen)
    s = torch.full((N,), 0.01, dtype=torch.float32, device="cuda")
    return w, s, N * K + N * 4


def graph_time(torch, calls, reps=20):
    """Capture the calls once into a CUDA graph, replay `reps` times; median ms
    per replay (CUDA events on the current stream)."""
    stream = torch.cuda.current_stream()
    for f in calls:
        f()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for f in calls:
            f()
    g.replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for e in ev:
        e[0].record(stream)
        g.replay()
        e[1].record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ev)


class WqStep:
    """The large weight-only projection (28672 x 5120) at one token, INT4 and
    e4m3, cycled over 8 weight copies larger than L2 (one step = the 8
    products in one CUDA graph)."""
    name = "wq_large_m1"

    def __init__(self, torch, kvq, seed, N=28672, K=5120, copies=8):
        self.torch, self.kvq = torch, kvq
        gen = torch.Generator(device="cuda").manual_seed(seed)
        self.N, self.K = N, K
        self.mats = {wd: [wq_weights(torch, kvq, gen, wd, N, K) for _ in range(copies)]
                     for wd in (kvq.W_INT4, kvq.W_E4M3)}
        self.x = torch.randn((1, K), device="cuda", generator=gen).to(torch.bfloat16)
        self.ys = [torch.empty((1, N), dtype=torch.float32, device="cuda") for _ in range(copies)]
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def time(self, warmup, steps):
        torch, kvq = self.torch, self.kvq
        peak, _ = measured_hbm_peak()
        out = {"workload": f"weight-only projection {self.N} x {self.K}, one token, "
                           f"{len(self.ys)} weight copies per step (larger than L2; no flush)",
               "steps": steps}
        for wd, name in ((kvq.W_E4M3, "e4m3"), (kvq.W_INT4, "int4")):
            calls = [(lambda w=w, s=s, y=y: kvq.kvq_wq_gemm(wd, w, s, self.x, y, err_word=self.err))
                     for (w, s, _), y in zip(self.mats[wd], self.ys)]
            ms = graph_time(torch, calls, max(steps, 3))
            nbytes = sum(m[2] for m in self.mats[wd])
            gbs = nbytes / (ms * 1e-3) / 1e9
            out[name] = {"us_per_product": round(ms * 1e3 / len(calls), 2),
                         "GBs": round(gbs, 1), "frac_of_measured_peak": round(gbs / peak, 4),
                         "bytes_per_product": nbytes // len(calls)}
        if int(self.err.item()) != 0:
            raise RuntimeError(f"device error bits {int(self.err.item()):#x}")
        out["int4_speedup_vs_e4m3"] = round(out["e4m3"]["us_per_product"]
                                            / out["int4"]["us_per_product"], 3)
        return out


def run_wq(args):
    """Weight-only INT4 vs e4m3 decode matrix products (kvq_wq_gemm), the
    pages' second decode workload: every generated token streams all the
    weights.  Per M (tokens in flight): (a) one decode step's projections of a
    40-layer stack of GLM-like shapes (distinct weights, 812 MB INT4 / 1.6 GB
    e4m3: larger than L2), captured as one CUDA graph and replayed; (b) one
    large projection (28672 x 5120) cycled over 8 weight copies.  Weights and
    activations are seeded random data (no trained weights); each product's
    output is discarded, so this times weight streaming, not a model."""
    import torch
    from fp8_paged_kv_attn_gb300 import kvq

    kvq.load()
    peak, _ = measured_hbm_peak()
    gen = torch.Generator(device="cuda").manual_seed(args.seed)

    kinds = ("stack", "large") if args.wq_kind == "all" else (args.wq_kind,)
    formats = [(kvq.W_E4M3, "e4m3"), (kvq.W_INT4, "int4")]
    if args.wq_w != "both":
        formats = [f for f in formats if f[1] == args.wq_w]
    ms_list = (args.wq_m,) if args.wq_m else (1, 8, 16, 32, 64)
    for kind in kinds:
        res = {}
        for wdtype, name in formats:
            if kind == "stack":
                mats = [wq_weights(torch, kvq, gen, wdtype, N, K) + (N, K)
                        for _ in range(WQ_LAYERS) for _, N, K in WQ_LAYER]
            else:
                mats = [wq_weights(torch, kvq, gen, wdtype, 28672, 5120) + (28672, 5120)
                        for _ in range(8)]
            nbytes = sum(m[2] for m in mats)
            for M in ms_list:
                xs = {K: torch.randn((M, K), device="cuda", generator=gen).to(torch.bfloat16)
                      for K in {m[4] for m in mats}}
                ys = [torch.empty((M, m[3]), dtype=torch.float32, device="cuda") for m in mats]
                calls = [(lambda m=m, y=y: kvq.kvq_wq_gemm(wdtype, m[0], m[1], xs[m[4]], y))
                         for m, y in zip(mats, ys)]
                ms = graph_time(torch, calls)
                gbs = nbytes / (ms * 1e-3) / 1e9
                res[(name, M)] = ms
                line = {"workload": f"wq_{kind}", "w": name, "M": M, "products": len(mats),
                        "weight_bytes": nbytes, "ms_per_step": round(ms, 4),
                        "tokens_per_s": round(M / (ms * 1e-3), 1), "GBs": round(gbs, 1),
                        "frac_of_measured_peak": round(gbs / peak, 4),
                        "flops_TFs": round(2.0 * M * sum(m[3] * m[4] for m in mats) /
                                           (ms * 1e-3) / 1e12, 1)}
                if name == "int4" and ("e4m3", M) in res:
                    line["speedup_vs_e4m3"] = round(res[("e4m3", M)] / ms, 3)
                print(json.dumps(line), flush=True)
            del mats


def main():
    args = parse_args()
    if args.workload == "wq":
        run_wq(args)
        return
    if args.workload == "pages":
        run_pages(args)
        return
    if args.workload == "prefill":
        run_prefill(args)
        return
    if args.workload == "handoff":
        run_handoff(args)
        return
    if args.workload:
        run_workload(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.impl == "reference":
        # the CPU oracle runs on rank 0 only; other ranks exit without work
        if int(os.environ.get("RANK", "0")) == 0:
            print(json.dumps(run_reference(args, 0)), flush=True)
        return
    dist, rank, world, local = dist_setup()
    result = run_gpu(args, dist, rank, world, local)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
