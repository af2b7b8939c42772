"""Benchmark of one decode step of hierarchically pruned, block-sparse attention over an
int8-keyed paged KV cache (append, query quantisation + int8 scoring, two pruning modules,
split-K attention + log-sum-exp merge), against the in-run dense bf16 decode kernel.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

Prints ONE JSON line (rank 0). Timing: the whole step (hsa_decode_step on device buffers)
is captured 10 times back to back in one CUDA graph, two replicas of the whole cache
alternating, so each step reads data the previous step did not touch (146 MB per step at
128K tokens, more than the 129 MB L2); the timed region replays it until K steps have run,
with one pair of CUDA events around all of them on the launching stream. The dense decode
and each kernel of the per-kernel breakdown (the scorer's roofline) are timed the same way,
from graphs of 10 back-to-back launches. `step_latency_us` is one step per graph replay with
events around each replay, which includes the graph launch. `--impl reference` times the CPU oracle on the
host cores instead.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse decode-attn µs/step & achieved HBM GB/s at 128K/1M ctx vs dense decode"
DEFAULT_CONFIG = "llama3-8b-128k"
EXTRA_CONFIG = "llama3-8b-1m"
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ ranks

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int) -> float:
    """Max of a float over all ranks (the value itself when world == 1)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def job_value(step_ms_max: float, world: int) -> float:
    """µs per decode step of the job: every rank runs its own independent decode problem, so
    a step of the job takes the slowest rank's step time (a latency; N replicas do not make
    a step faster)."""
    return step_ms_max * 1e3


def job_steps_per_s(step_ms_max: float, world: int) -> float:
    """Aggregate decode steps per second of the whole job: N independent replicas complete N
    steps in the slowest rank's step time."""
    return world / (step_ms_max * 1e-3)


# ------------------------------------------------------------ measurement

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed loop runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.2)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def traffic_record(kernel_file: str, summary_name: str):
    """DRAM bytes per launch recorded in a committed ncu summary, valid only while the
    kernel source it was measured on is unchanged (matched by sha256)."""
    path = os.path.join(ROOT, "profiles", summary_name)
    src = os.path.join(ROOT, "kv_cache_int8_gb300", "csrc", kernel_file)
    try:
        text = open(path, encoding="utf-8").read()
        want = re.search(r"source_sha256:\s*([0-9a-f]{64})", text).group(1)
        bytes_ = float(re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text).group(1))
    except Exception:
        return None
    have = hashlib.sha256(open(src, "rb").read()).hexdigest()
    return bytes_ if have == want else None


# -------------------------------------------------------------- GPU arm

class Case:
    """One workload resident on the GPU: cache replicas (two, or five when one replica's key
    codes are smaller than L2), their int8 codes and scales, buffers, and the captured
    graphs."""

    KERNELS = ("step", "append", "score", "prune", "attend", "dense")
    BURST = 10  # a multiple of every replica count
    L2_BYTES = 129_000_000  # GB300: 129 MB
    REFRESH = 4
    CACHE_SLOTS = 8192  # GPU block cache of the offloaded case: 64 MiB of K/V blocks

    def __init__(self, name: str, seed: int, device, dense: bool = True):
        import torch
        from kv_cache_int8_gb300 import hsa
        from kv_cache_int8_gb300 import workloads as W
        self.torch, self.hsa = torch, hsa
        self.cfg = W.CONFIGS[name]
        cfg = self.cfg
        self.kernels = self.KERNELS if dense else tuple(k for k in self.KERNELS if k != "dense")
        if cfg.kv_on_host:  # the step and the attention through the GPU block cache too
            self.kernels = self.kernels + ("step_cached", "attend_cached", "step_cached_mass")
        # offloaded K/V: one pinned host copy (both "replicas" alias it; steps are separated by
        # an L2 flush instead, see timed_steps)
        wl = W.make_workload(cfg, seed=seed, device=str(device), host_pinned=cfg.kv_on_host)
        self.wl = wl
        self.flush = None
        if cfg.kv_on_host:
            self.flush = torch.empty(512 << 20, dtype=torch.uint8, device=device)
        self.d = hsa.Dims(batch=cfg.batch, hq=cfg.hq, hkv=cfg.hkv,
                          max_pages_per_seq=wl["max_pages"], num_pages=wl["num_pages"],
                          chunk=cfg.chunk, k1=cfg.k1, k2=cfg.k2, sink=cfg.sink,
                          window=cfg.window, kv_on_host=cfg.kv_on_host, chunk0=cfg.chunk0,
                          k0=cfg.k0, key_bits=cfg.key_bits, per_head=cfg.per_head,
                          key_fp8=cfg.key_fp8)
        d = self.d
        R = cfg.hq if cfg.per_head else cfg.hkv  # selection rows per sequence
        B, Hq, Hkv = cfg.batch, cfg.hq, cfg.hkv
        self.q = wl["q"]
        self.pt, self.lens = wl["page_table"], wl["seq_lens"]
        # replicas: consecutive steps read different ones; two when one replica's key codes
        # (the scan of a step) exceed L2, else five, so that between two reads of the same
        # codes the steps read several times L2 of other data (4-bit codes at 128K tokens,
        # 67 MB a replica)
        kq_shape = list(wl["k_cache"].shape)
        kq_shape[-1] = kq_shape[-1] * cfg.key_bits // 8  # 4-bit codes: two per byte
        codes = cfg.hkv * sum(wl["lens"]) * 128 * cfg.key_bits // 8
        self.nrep = 2 if cfg.kv_on_host or codes >= self.L2_BYTES else 5
        if cfg.kv_on_host:
            self.k = [wl["k_cache"], wl["k_cache"]]
            self.v = [wl["v_cache"], wl["v_cache"]]
        else:
            self.k = [wl["k_cache"]] + [wl["k_cache"].clone() for _ in range(self.nrep - 1)]
            self.v = [wl["v_cache"]] + [wl["v_cache"].clone() for _ in range(self.nrep - 1)]
        self.kq = [torch.zeros(kq_shape, dtype=torch.int8, device=device)
                   for _ in range(self.nrep)]
        self.ks = [torch.zeros((B, Hkv, 128), dtype=torch.float32, device=device)
                   for _ in range(self.nrep)]
        wq = hsa.workspace(d, hsa.HSA_OP_QUANTIZE)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        hsa.hsa_quantize_keys(d, self.k[0], self.pt, self.lens, 0, 0, self.kq[0], self.ks[0], wq)
        e1.record()
        for r in range(1, self.nrep):
            hsa.hsa_quantize_keys(d, self.k[r], self.pt, self.lens, 0, 0, self.kq[r], self.ks[r],
                                  wq)
        torch.cuda.synchronize()
        self.quantize_ms = e0.elapsed_time(e1)
        # the new token of the step: re-append the current last token (cache unchanged)
        lens = wl["lens"]
        ptc = wl["page_table"].cpu()
        kdev = self.k[0].device
        pages = torch.tensor([int(ptc[b, (n - 1) // 16]) for b, n in enumerate(lens)],
                             device=kdev)
        slots = torch.tensor([(n - 1) % 16 for n in lens], device=kdev)
        self.k_new = self.k[0][pages, :, slots].contiguous().to(device)
        self.v_new = self.v[0][pages, :, slots].contiguous().to(device)
        self.ws_sel = hsa.workspace(d, hsa.HSA_OP_SELECT)
        self.ws_att = hsa.workspace(d, hsa.HSA_OP_ATTEND)
        self.ws_den = hsa.workspace(d, hsa.HSA_OP_DENSE)
        self.ws_step = hsa.workspace(d, hsa.HSA_OP_STEP)
        if cfg.kv_on_host:
            self.cache_capacity = self.CACHE_SLOTS
            self.cache = hsa.block_cache(d, self.cache_capacity)
            self.ws_cached = hsa.workspace(d, hsa.HSA_OP_CACHED)
            # the same cache under the cumulative-attention-mass eviction policy
            self.d_mass = dataclasses.replace(d, cache_policy=1)
            self.cache_mass = hsa.block_cache(self.d_mass, self.cache_capacity)
            self.ws_step_mass = hsa.workspace(self.d_mass, hsa.HSA_OP_STEP)
        self.bm = torch.zeros((B, R, d.max_pages_per_seq), dtype=torch.int32, device=device)
        self.tm = torch.zeros((B, R, (d.max_pages_per_seq + 3) // 4), dtype=torch.int32,
                              device=device)
        self.chunk_idx = torch.zeros((B, R, max(d.k1, 1)), dtype=torch.int32, device=device)
        self.n_chunks = torch.zeros((B, R), dtype=torch.int32, device=device)
        self.block_idx = torch.zeros((B, R, max(d.k2, 1)), dtype=torch.int32, device=device)
        self.n_blocks = torch.zeros((B, R), dtype=torch.int32, device=device)
        self.out = torch.zeros((B, Hq, 128), dtype=torch.float32, device=device)
        self.lse = torch.zeros((B, Hq), dtype=torch.float32, device=device)
        self.out_d = torch.zeros_like(self.out)
        self.lse_d = torch.zeros_like(self.lse)

    # the whole step, the pruning form's four kernels one at a time (the per-kernel
    # breakdown), and the dense comparison, on replica r
    def step(self, r):
        self.hsa.hsa_decode_step(self.d, self.q, self.k_new, self.v_new, self.out, self.lse,
                                 self.k[r], self.v[r], self.kq[r], self.ks[r], self.pt,
                                 self.lens, self.block_idx, self.n_blocks, self.ws_step)

    def step_cached(self, r):
        self.hsa.hsa_decode_step_cached(self.d, self.q, self.k_new, self.v_new, self.out,
                                        self.lse, self.k[r], self.v[r], self.kq[r], self.ks[r],
                                        self.pt, self.lens, self.block_idx, self.n_blocks,
                                        self.cache, self.cache_capacity, self.ws_step)

    def step_cached_mass(self, r):
        self.hsa.hsa_decode_step_cached(self.d_mass, self.q, self.k_new, self.v_new, self.out,
                                        self.lse, self.k[r], self.v[r], self.kq[r], self.ks[r],
                                        self.pt, self.lens, self.block_idx, self.n_blocks,
                                        self.cache_mass, self.cache_capacity, self.ws_step_mass)

    def attend_cached(self, r):
        self.hsa.hsa_attend_cached(self.d, self.q, self.k[r], self.v[r], self.pt, self.lens,
                                   self.block_idx, self.n_blocks, self.cache,
                                   self.cache_capacity, self.out, self.lse, self.ws_cached)

    def reuse(self, r):
        """A step that reuses the last whole step's selection (append + attend)."""
        self.hsa.hsa_decode_step_reuse(self.d, self.q, self.k_new, self.v_new, self.out,
                                       self.lse, self.k[r], self.v[r], self.kq[r], self.ks[r],
                                       self.pt, self.lens, self.block_idx, self.n_blocks,
                                       self.ws_step)

    def append(self, r):
        self.hsa.hsa_append_kv(self.d, self.k_new, self.v_new, self.k[r], self.v[r], self.kq[r],
                               self.ks[r], self.pt, self.lens)

    def score(self, r):
        self.hsa.hsa_score_blocks(self.d, self.q, self.kq[r], self.ks[r], self.pt, self.lens,
                                  self.bm, self.tm)

    def prune(self, r):
        self.hsa.hsa_prune(self.d, self.lens, self.bm, self.tm, self.chunk_idx, self.n_chunks,
                           self.block_idx, self.n_blocks)

    def attend(self, r):
        self.hsa.hsa_attend(self.d, self.q, self.k[r], self.v[r], self.pt, self.lens,
                            self.block_idx, self.n_blocks, self.out, self.lse, self.ws_att)

    def dense(self, r):
        self.hsa.dense_decode(self.d, self.q, self.k[r], self.v[r], self.pt, self.lens,
                              self.out_d, self.lse_d, self.ws_den)

    def capture(self):
        torch = self.torch
        self.graphs = {}
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for r in range(self.nrep):
                for name in self.kernels:
                    getattr(self, name)(r)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        for r in range(self.nrep):
            for name in self.kernels:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    getattr(self, name)(r)
                self.graphs[(name, r)] = g
        # the decode loop: a whole step, then REFRESH - 1 steps reusing its selection
        for r in range(self.nrep):
            self.step(r)
            self.reuse(r)
        torch.cuda.synchronize()
        for r in range(self.nrep):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.step(r)
                for _ in range(self.REFRESH - 1):
                    self.reuse(r)
            self.graphs[("loop", r)] = g
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.reuse(r)
            self.graphs[("reuse", r)] = g
        # per-kernel durations: BURST launches of one kernel in one graph, replicas
        # alternating (so that every launch of the scan reads data the previous one did not)
        self.burst = {}
        if self.flush is None:
            for name in self.kernels:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for i in range(self.BURST):
                        getattr(self, name)(i % self.nrep)
                self.burst[name] = g
        torch.cuda.synchronize()

    # ---- algorithmic bytes (what the method must move; see the design notes)
    def candidate_tokens(self):
        c = self.cfg
        return sum(max(0, n - c.window - c.sink) for n in self.wl["lens"])

    def attended_tokens(self):
        """|T| summed over (sequence, selection row): sink + window + the kept blocks'
        candidate tokens, from the selection of the last step. A row is a kv head, or a
        query head with per-head selection (whose K/V are then read once per query head)."""
        c = self.cfg
        nb = self.n_blocks.cpu()
        bi = self.block_idx.cpu()
        total = 0
        for b, n in enumerate(self.wl["lens"]):
            sink_end = min(c.sink, n)
            w0 = max(n - c.window, sink_end)
            base = sink_end + (n - w0)
            for h in range(nb.shape[1]):
                total += base
                for k in bi[b, h, : int(nb[b, h])].tolist():
                    total += max(0, min(16 * k + 16, n - c.window) - max(16 * k, c.sink))
        return total

    def bytes_score(self):
        c = self.cfg
        blocks = sum(max(0, -(-(n - c.window) // 16) - c.sink // 16) for n in self.wl["lens"])
        return (c.hkv * self.candidate_tokens() * 128 * c.key_bits // 8 + c.batch * c.hq * 128 * 2 +
                c.batch * c.hkv * 128 * 4 + self.bm.shape[1] * blocks * 4)

    def bytes_attend(self):
        c = self.cfg
        return (self.attended_tokens() * 128 * 2 * 2 + c.batch * c.hq * 128 * 2 +
                c.batch * c.hq * 129 * 4)

    def bytes_dense(self):
        c = self.cfg
        return (c.hkv * sum(self.wl["lens"]) * 128 * 2 * 2 + c.batch * c.hq * 128 * 2 +
                c.batch * c.hq * 129 * 4)


def timed_steps(case, steps: int, names, sampler=None):
    """Replay the graphs of `names` for `steps` steps, alternating replicas, with events
    around each replay. Returns per-name mean ms and per-step mean ms."""
    torch = case.torch
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
           for _ in range(steps)]
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    # a short head start so that the launch queue runs ahead of the GPU
    torch.cuda._sleep(2_000_000)
    for i in range(steps):
        r = i % case.nrep
        ev = evs[i]
        if case.flush is not None:
            case.flush.fill_(i & 0xFF)  # evict the previous step's data from L2
        ev[0].record()
        for j, name in enumerate(names):
            case.graphs[(name, r)].replay()
            ev[j + 1].record()
    torch.cuda.synchronize()
    if sampler:
        sampler.stop()
    per = {name: statistics.fmean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(steps))
           for j, name in enumerate(names)}
    step = statistics.fmean(evs[i][0].elapsed_time(evs[i][-1]) for i in range(steps))
    return per, step


def timed_step_run(case, steps: int, sampler=None):
    """The timed region: `steps` whole steps back to back, as replays of the graph of BURST
    steps (cache replicas alternating inside it) plus one graph for the remainder, with one
    pair of CUDA events around all of them. Returns ms per step. The 3M offloaded case, whose
    steps need an L2-evicting write between them, is timed one replay per step instead."""
    torch = case.torch
    if "step" not in case.burst:
        _, step = timed_steps(case, steps, ("step",), sampler)
        return step
    whole, rest = divmod(steps, case.BURST)
    tail = None
    if rest:
        tail = torch.cuda.CUDAGraph()
        with torch.cuda.graph(tail):
            for i in range(rest):
                case.step(i % case.nrep)
        tail.replay()
    case.burst["step"].replay()  # untimed: the burst graph's first replay
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    torch.cuda._sleep(2_000_000)  # a head start so that the launch queue runs ahead of the GPU
    e0.record()
    for _ in range(whole):
        case.burst["step"].replay()
    if tail is not None:
        tail.replay()
    e1.record()
    torch.cuda.synchronize()
    if sampler:
        sampler.stop()
    return e0.elapsed_time(e1) / steps


def host_link_copy_gbs(device, mib: int = 512) -> float:
    """Pinned host -> device copy-engine rate (GB/s): the host link's measured read rate, the
    denominator for kernels that read K/V from mapped host memory."""
    import torch
    h = torch.empty(mib << 20, dtype=torch.uint8).pin_memory()
    d = torch.empty(mib << 20, dtype=torch.uint8, device=device)
    d.copy_(h, non_blocking=True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(3):
        d.copy_(h, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    return 3 * (mib << 20) / (e0.elapsed_time(e1) * 1e6)


def burst_times(case, names, reps: int):
    """Average duration of one launch of each kernel: `reps` replays of its burst graph
    (BURST launches back to back) with CUDA events around each replay, after 3 warm-up
    replays; falls back to one-launch graphs (timed_steps) when there are no bursts."""
    torch = case.torch
    if not case.burst:
        timed_steps(case, 3, names)
        per, _ = timed_steps(case, reps, names)
        return per
    out = {}
    for name in names:
        g = case.burst[name]
        for _ in range(3):
            g.replay()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        torch.cuda.synchronize()
        torch.cuda._sleep(2_000_000)
        for a, b in evs:
            a.record()
            g.replay()
            b.record()
        torch.cuda.synchronize()
        out[name] = statistics.fmean(a.elapsed_time(b) for a, b in evs) / case.BURST
    return out


def e2e_steps(case, steps: int):
    """The public whole-step call with pinned host inputs and outputs, timed by the host
    clock (time.perf_counter) around the call and the stream's synchronisation, per step:
    the plain call through the binding (every argument marshalled, the kernels launched one
    by one), and its decode-loop form hsa.DecodeStep (arguments marshalled once, the step
    replayed from the CUDA graph it records on its first call), the latter also with CUDA
    events on the stream. Returns ({form: mean us}, h2d bytes, d2h bytes)."""
    torch, hsa = case.torch, case.hsa
    c = case.cfg
    q_h = case.q.cpu().pin_memory()
    kn_h = case.k_new.cpu().pin_memory()
    vn_h = case.v_new.cpu().pin_memory()
    out_h = torch.zeros((c.batch, c.hq, 128), dtype=torch.float32).pin_memory()
    lse_h = torch.zeros((c.batch, c.hq), dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream()

    def plain(r):
        hsa.hsa_decode_step(case.d, q_h, kn_h, vn_h, out_h, lse_h, case.k[r], case.v[r],
                            case.kq[r], case.ks[r], case.pt, case.lens, None, None, case.ws_step,
                            io_on_host=True)

    graphs = [hsa.DecodeStep(case.d, q_h, kn_h, vn_h, out_h, lse_h, case.k[r], case.v[r],
                             case.kq[r], case.ks[r], case.pt, case.lens, None, None,
                             case.ws_step, io_on_host=True, graph=True) for r in range(2)]

    def host_clock(fn):
        times = []
        for i in range(steps + 3):
            t0 = time.perf_counter()
            fn(i & 1)
            stream.synchronize()
            t1 = time.perf_counter()
            if i >= 3:
                times.append((t1 - t0) * 1e6)
        return statistics.fmean(times)

    res = {"plain_call_us": host_clock(plain), "decode_step_graph_us": host_clock(lambda r: graphs[r]())}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev = []
    for i in range(steps + 3):
        e0.record()
        graphs[i & 1]()
        e1.record()
        e1.synchronize()
        if i >= 3:
            ev.append(e0.elapsed_time(e1) * 1e3)
    res["decode_step_graph_events_us"] = statistics.fmean(ev)
    h2d = q_h.numel() * 2 + kn_h.numel() * 2 + vn_h.numel() * 2
    d2h = out_h.numel() * 4 + lse_h.numel() * 4
    return res, h2d, d2h


def gpu_case_numbers(name, seed, device, steps, warmup, sampler, peak, world=1, dense=True):
    import torch
    from kv_cache_int8_gb300 import hsa
    case = Case(name, seed, device, dense)
    case.capture()
    names = ("append", "score", "prune", "attend")
    # the timed region: K whole steps back to back
    timed_steps(case, max(3, warmup), ("step",))                   # warm-up
    barrier(world)
    step_ms = timed_step_run(case, steps, sampler)
    barrier(world)
    # the latency of one step launched on its own: one graph replay per step, events around
    # each (includes the graph launch)
    _, latency_ms = timed_steps(case, max(3, min(steps, 1000)), ("step",))
    # the decode loop (selection refreshed every REFRESH steps) and the reuse step alone
    lsteps = max(3, min(steps // case.REFRESH, 500))
    timed_steps(case, 3, ("loop", "reuse"))
    lper, _ = timed_steps(case, lsteps, ("loop", "reuse"))
    cached = {}
    if getattr(case, "cache", None) is not None:
        names_c = ("step_cached", "attend_cached", "step_cached_mass")
        timed_steps(case, 3, names_c)
        cached, _ = timed_steps(case, max(3, min(steps, 300)), names_c)
    # kernel breakdown: the average launch duration of each of the pruning form's four
    # kernels (the scorer's is the roofline's)
    bsteps = max(3, min(steps // 10, 200))
    per = burst_times(case, names, bsteps)
    if dense:
        dper = burst_times(case, ("dense",), max(3, bsteps // 4))
    else:
        dper = {"dense": float("nan")}
    for w in (case.ws_step, case.ws_sel, case.ws_att, case.ws_den) + (
            (case.ws_cached, case.ws_step_mass) if getattr(case, "cache", None) is not None
            else ()):
        code = hsa.hsa_read_device_error(w)
        assert code == 0, f"device error word {code}"
    recall = torch.exp(case.lse.double() - case.lse_d.double())  # restriction identity
    if not dense:
        recall = torch.full_like(recall, float("nan"))
    sel_ms = per["score"] + per["prune"]
    res = {
        "case": case,
        "dims": case.d,
        "step_ms": step_ms,
        "latency_ms": latency_ms,
        "loop_step_ms": lper["loop"] / case.REFRESH,
        "reuse_step_ms": lper["reuse"],
        "cached_ms": cached,
        "per_ms": per,
        "select_ms": sel_ms,
        "dense_ms": dper["dense"],
        "bytes": {"score": case.bytes_score(), "attend": case.bytes_attend(),
                  "dense": case.bytes_dense()},
        "recall": {"mean": float(recall.mean()), "min": float(recall.min())},
        "quantize_ms": case.quantize_ms,
        "replicas": case.nrep,
    }
    b = res["bytes"]
    res["gbs"] = {
        "score": b["score"] / (per["score"] * 1e6),
        "select": b["score"] / (sel_ms * 1e6),
        "attend": b["attend"] / (per["attend"] * 1e6),
        "dense": b["dense"] / (dper["dense"] * 1e6),
        "step": (b["score"] + b["attend"]) / (step_ms * 1e6),
    }
    res["frac"] = {k: v / peak for k, v in res["gbs"].items()}
    return res


# ------------------------------------------------------------- CPU oracle

def oracle_step_sample(name: str, seed: int, budget_s: float, max_samples: int,
                       warmup: int = 0, one_thread: bool = True):
    """Time the CPU oracle's per-step work (append codes, query codes + scoring + both
    modules, sparse attention): whole steps, the oracle's OpenMP loops spreading each
    (sequence, kv head) pair's token blocks (scoring) and the pairs (attention) over the
    host cores, until `budget_s` seconds or `max_samples` steps, after `warmup` untimed
    steps; then one pair at a time on one thread, once per pair, scaled to a whole step.
    Returns (µs per whole step on the cores, steps, threads used, description, µs per whole
    step on one thread)."""
    import numpy as np
    import oracle
    from kv_cache_int8_gb300 import workloads as W
    cfg = W.CONFIGS[name]
    gen_dev = "cpu"
    if cfg.context is None or cfg.context > (1 << 17):  # large inputs: drawn on the GPU
        import torch
        gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    wl = W.make_workload(cfg, seed=seed, device=gen_dev)
    if gen_dev != "cpu":
        wl = {k: (v.cpu() if hasattr(v, "cpu") else v) for k, v in wl.items()}
        import torch
        torch.cuda.empty_cache()
    od = oracle.Dims(batch=cfg.batch, hq=cfg.hq, hkv=cfg.hkv, head_dim=128, page_size=16,
                     max_pages_per_seq=wl["max_pages"], num_pages=wl["num_pages"],
                     chunk=cfg.chunk, block=16, k1=cfg.k1, k2=cfg.k2, sink=cfg.sink,
                     window=cfg.window, chunk0=cfg.chunk0, k0=cfg.k0, key_bits=cfg.key_bits,
                     per_head=cfg.per_head, key_fp8=cfg.key_fp8)
    q, k, v = (W.to_numpy_bits(wl[x]) for x in ("q", "k_cache", "v_cache"))
    pt, lens = wl["page_table"].numpy(), wl["seq_lens"].numpy()
    kq, sc = oracle.quantize_keys(od, k, pt, lens)             # cache state, not per step
    pairs = [(b, h) for b in range(cfg.batch) for h in range(cfg.hkv)]
    G = cfg.hq // cfg.hkv

    def step(bh=None, qh=None):
        oracle.quantize_append(od, k, pt, lens, -1, sc, kq)
        sel = oracle.select(od, q, sc, kq, pt, lens, bh_mask=bh)
        oracle.attend(od, q, k, v, pt, lens, sel["block_idx"], sel["n_blocks"], qh_mask=qh)

    for _ in range(warmup):  # untimed: pages in the inputs and the oracle's code
        step()
    t_total, n = 0.0, 0
    start = time.perf_counter()
    while n < max_samples and (time.perf_counter() - start) < budget_s:
        t0 = time.perf_counter()
        step()
        t_total += time.perf_counter() - t0
        n += 1
    us_step = t_total / max(n, 1) * 1e6
    threads = oracle.num_threads()
    # one thread: each pair once
    t1 = 0.0
    if one_thread:
        oracle.set_num_threads(1)
    for b, h in (pairs if one_thread else ()):
        bh = np.zeros((cfg.batch, cfg.hkv), dtype=np.int32)
        bh[b, h] = 1
        qh = np.zeros((cfg.batch, cfg.hq), dtype=np.int32)
        qh[b, h * G:(h + 1) * G] = 1
        t0 = time.perf_counter()
        step(bh, qh)
        t1 += time.perf_counter() - t0
    if one_thread:
        oracle.set_num_threads(threads)
    us_1 = t1 * 1e6
    desc = (f"{n} whole steps ({name}: append codes, query codes, int8 scoring of the whole "
            f"context, both modules, sparse attention), each of the {len(pairs)} (sequence, "
            f"kv head) pairs' token blocks spread over {threads} threads of the host's "
            f"{os.cpu_count()} cores"
            + (f"; one thread, pair by pair: {us_1 / 1e3:.1f} ms per step" if one_thread else ""))
    return us_step, n, threads, desc, us_1


def W_CONFIGS():
    from kv_cache_int8_gb300 import workloads as W
    return W.CONFIGS


# ------------------------------------------------------------------ main

def run_reference(args, world, rank):
    if rank != 0:
        return 0
    from kv_cache_int8_gb300 import workloads as W
    budget = float(os.environ.get("HSA_REF_BUDGET_S", "20"))
    us, n, cores, desc, us_1 = oracle_step_sample(args.config, 0, budget, max(1, args.steps),
                                                  warmup=args.warmup)
    line = {
        "metric": METRIC, "value": us, "unit": "us/step", "n_gpus": args.gpus,
        "steps": n, "steps_requested": args.steps, "warmup": args.warmup,
        "ms_per_step": us / 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "int8+f64",
        "data": "synthetic (seeded)", "impl": "reference",
        "config": {"workload": workload_text(W.CONFIGS[args.config])},
        "cpu_baseline": {"value": us, "unit": "us/step", "cores": cores, "kind": "oracle",
                         "sample": desc, "one_thread_us": us_1},
        "e2e": {"value": us, "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def profile_steps(name, device, steps, warmup):
    """Direct launches of the whole step (and of dense decode) for a profiler's launch list:
    `warmup` steps, then `steps` steps and steps // 2 dense decodes, replicas alternating
    (no dense decode when K/V live in host memory)."""
    import torch
    case = Case(name, 0, device, dense=not W_CONFIGS()[name].kv_on_host)
    for i in range(warmup):
        case.step(i % case.nrep)
    torch.cuda.synchronize()
    for i in range(steps):
        case.step(i % case.nrep)
    n_dense = steps // 2 if "dense" in case.kernels else 0
    for i in range(n_dense):
        case.dense(i % case.nrep)
    torch.cuda.synchronize()
    for w in (case.ws_step, case.ws_den):
        code = case.hsa.hsa_read_device_error(w)
        assert code == 0, f"device error word {code}"
    print(f"profiled {steps} steps and {n_dense} dense decodes of {name}")
    return 0


def workload_text(cfg):
    mod0 = f"chunk0 {cfg.chunk0} keep K0 {cfg.k0}, " if cfg.k0 > 0 else ""
    return (f"{cfg.name}: batch {cfg.batch}, Hq {cfg.hq}, Hkv {cfg.hkv}, d 128, context "
            f"{cfg.context}, {mod0}chunk {cfg.chunk} keep K1 {cfg.k1}, block 16 keep K2 "
            f"{cfg.k2}, sink {cfg.sink}, window {cfg.window}; bf16 K/V in 16-token pages, "
            + ("FP8 E4M3" if cfg.key_fp8 else f"int{cfg.key_bits}") + " per-channel keys"
            + ("; per-head selection" if cfg.per_head else ""))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=6000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extra", action="store_true", help="skip the 1M-token extra case")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--profile-steps", type=int, default=0,
                    help="for profilers: run this many whole steps with direct launches (no "
                         "CUDA graphs), then half as many dense decodes, and exit")
    args = ap.parse_args()
    world, rank, local = dist_env()

    if args.impl == "reference":
        return run_reference(args, world, rank)

    import torch
    import __graft_entry__ as entry
    from kv_cache_int8_gb300 import workloads as W
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    entry.build()
    device = torch.device("cuda", torch.cuda.current_device())
    peak, peak_kind = peaks()
    sampler = ClockSampler(local) if rank == 0 else None

    if args.profile_steps > 0:
        return profile_steps(args.config, device, args.profile_steps, args.warmup)

    main_res = gpu_case_numbers(args.config, rank, device, args.steps, args.warmup, sampler, peak,
                                world)
    case = main_res["case"]
    step_ms = reduce_max(main_res["step_ms"], world)
    e2e, h2d, d2h = (None, 0, 0)
    if not args.no_e2e:
        e2e, h2d, d2h = e2e_steps(case, min(args.steps, 1000))
        e2e = {k: reduce_max(v, world) for k, v in e2e.items()}
    clocks = sampler.summary() if sampler else None
    del case, main_res["case"]
    torch.cuda.empty_cache()

    extra = {}
    if not args.no_extra:
        # the batched paged configuration and the 3M-token offloaded one (K/V in pinned host
        # memory, read over the host link by the attend kernel)
        for name, dense in (("paged-b8-32k-128k", True), ("llama3-8b-3m-offload", False),
                            ("llama3-8b-1m-3mod", True), ("llama3-8b-128k-int4", True),
                            ("llama3-8b-1m-int4", True), ("llama3-70b-128k", True),
                            ("llama3-8b-128k-perhead", True), ("llama3-8b-128k-fp8", True)):
            r = gpu_case_numbers(name, rank, device, min(args.steps, 500), args.warmup, None,
                                 peak, world, dense=dense)
            del r["case"]
            torch.cuda.empty_cache()
            extra[name] = {
                "us_per_step": r["step_ms"] * 1e3, "step_latency_us": r["latency_ms"] * 1e3,
                "score_us": r["per_ms"]["score"] * 1e3,
                **({"host_link_copy_gbs": host_link_copy_gbs(device),
                    "us_per_step_block_cache": r["cached_ms"]["step_cached"] * 1e3,
                    "attend_block_cache_us": r["cached_ms"]["attend_cached"] * 1e3,
                    "us_per_step_block_cache_mass_policy": r["cached_ms"]["step_cached_mass"] * 1e3,
                    "block_cache_slots": Case.CACHE_SLOTS} if r["cached_ms"] else {}),
                "prune_us": r["per_ms"]["prune"] * 1e3, "attend_us": r["per_ms"]["attend"] * 1e3,
                "dense_us": r["dense_ms"] * 1e3 if dense else None,
                "recall_vs_dense": r["recall"] if dense else None,
                "score_gbs": r["gbs"]["score"],
                "attend_gbs" + ("_host_link" if r["cached_ms"] else ""): r["gbs"]["attend"],
                "bytes": r["bytes"], "quantize_keys_ms": r["quantize_ms"],
                "replicas": r["replicas"],
            }
    if not args.no_extra and args.config != EXTRA_CONFIG:
        r = gpu_case_numbers(EXTRA_CONFIG, rank, device, min(args.steps, 1500), args.warmup, None,
                             peak, world)
        del r["case"]
        torch.cuda.empty_cache()
        extra[EXTRA_CONFIG] = {
            "us_per_step": r["step_ms"] * 1e3, "step_latency_us": r["latency_ms"] * 1e3,
            "select_us": r["select_ms"] * 1e3, "score_us": r["per_ms"]["score"] * 1e3,
            "prune_us": r["per_ms"]["prune"] * 1e3, "attend_us": r["per_ms"]["attend"] * 1e3,
            "dense_us": r["dense_ms"] * 1e3,
            "speedup_vs_dense": r["dense_ms"] / r["step_ms"],
            "gbs": r["gbs"], "frac_of_peak": r["frac"], "bytes": r["bytes"],
            "recall_vs_dense": r["recall"], "quantize_keys_ms": r["quantize_ms"],
        }

    barrier(world)
    if rank != 0:
        return 0

    cpu = None
    if not args.no_cpu_baseline:
        us, n, cores, desc, us_1 = oracle_step_sample(args.config, 0, 15.0, 10 ** 9, warmup=1)
        cpu = {"value": us, "unit": "us/step", "cores": cores, "host_cores": os.cpu_count(),
               "kind": "oracle", "sample": desc, "one_thread_us": us_1, "per_config": {}}
        # the oracle on the other headline configurations, a few steps each
        for name in (() if args.no_extra else (EXTRA_CONFIG, "paged-b8-32k-128k")):
            if name == args.config:
                continue
            us_c, n_c, cores_c, desc_c, _ = oracle_step_sample(name, 0, 4.0, 10 ** 9,
                                                               warmup=1, one_thread=False)
            cpu["per_config"][name] = {"value": us_c, "unit": "us/step", "steps": n_c,
                                       "cores": cores_c, "sample": desc_c}

    per = main_res["per_ms"]
    from kv_cache_int8_gb300 import hsa as hsa_mod
    d0 = main_res["dims"]
    kernels_per_step = hsa_mod.hsa_decode_step_kernels(d0)
    traffic = traffic_record("score.cu", "score_blocks_llama3-8b-128k.md")
    cfg = W.CONFIGS[args.config]
    line = {
        "metric": METRIC,
        "value": job_value(step_ms, world),
        "job_steps_per_s": job_steps_per_s(step_ms, world),
        "unit": "us/step",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_ms,
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int8+fp32",
        "data": "synthetic (seeded workload generator; N(0,1) bf16 K/V, 4 x8 outlier key "
                "channels, 8 planted keys per kv head)",
        "config": {
            "workload": workload_text(cfg),
            "step": "append new token + int8 scoring + 2 pruning modules + split-K attention "
                    f"(hsa_decode_step: {kernels_per_step} kernels: the scorer, which also "
                    "appends the token and records each row's range of maxima, and the "
                    "attention, which runs both pruning modules itself; steps replayed from "
                    "CUDA graphs)" if kernels_per_step == 2 else
                    f"append new token + int8 scoring + 2 pruning modules + split-K attention "
                    f"(hsa_decode_step: {kernels_per_step} kernels, CUDA graphs)",
            "l2": "2 cache replicas alternate: every step reads data the previous step did not "
                  "touch (more than the 129 MB L2)",
            "parallelism": f"replicas x{world} (independent decode problems per GPU)",
        },
        "roofline": {
            "bound": "hbm",
            "kernel": "score_blocks (int8 scan of every candidate key)",
            "achieved": main_res["gbs"]["score"],
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": main_res["frac"]["score"],
            "traffic": traffic,
            "algorithmic_bytes_per_launch": main_res["bytes"]["score"],
        },
        "cpu_baseline": cpu,
        "e2e": None if e2e is None else {
            "value": job_value(e2e["plain_call_us"] * 1e-3, world), "unit": "us/step",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "path": "hsa_decode_step called through the binding (ctypes, every argument "
                    "marshalled per call) with pinned host q/k_new/v_new/out/lse (mapped: a "
                    "kernel stages the inputs, the attention writes the outputs to host "
                    "memory; the two replica buffer sets alternate, and the library replays "
                    "the CUDA graph it recorded at the first call with each set); host clock "
                    "(time.perf_counter) around the call and the stream's synchronisation, "
                    "mean over steps",
            "decode_step_graph_us": e2e["decode_step_graph_us"],
            "decode_step_graph_events_us": e2e["decode_step_graph_events_us"],
            "forms": "decode_step_graph_us: hsa.DecodeStep (the decode-loop form: arguments "
                     "marshalled once, the step replayed from a CUDA graph), host clock; "
                     "decode_step_graph_events_us: the same with CUDA events on the stream"},
        "gpu_launches": kernels_per_step * args.steps,
        "timing": "value: K whole steps (hsa_decode_step with device buffers) back to back, "
                  "replayed from a CUDA graph of 10 steps (cache replicas alternating), one "
                  "pair of CUDA events around all K, the same method as the dense decode and "
                  "the per-kernel breakdown (graphs of 10 back-to-back launches of one kernel: "
                  "the pruning form's append, scorer, pruning kernel and attention, through "
                  "their own entry points; at 128K the step itself runs the scorer and the "
                  "selecting attention); step_latency_us: one step per graph replay, events "
                  "around each replay (includes the graph launch)",
        "step_latency_us": main_res["latency_ms"] * 1e3,
        "clocks": clocks,
        "breakdown_us": {k: v * 1e3 for k, v in per.items()},
        "select_us": main_res["select_ms"] * 1e3,
        "dense_us": main_res["dense_ms"] * 1e3,
        "speedup_vs_dense": main_res["dense_ms"] / step_ms,
        "decode_loop": {
            "refresh_every": Case.REFRESH,
            "us_per_step": main_res["loop_step_ms"] * 1e3,
            "reuse_step_us": main_res["reuse_step_ms"] * 1e3,
            "timing": "graph of one whole step + 3 steps reusing its selection, per step",
        },
        "gbs": main_res["gbs"],
        "frac_of_peak": main_res["frac"],
        "bytes": main_res["bytes"],
        "recall_vs_dense": main_res["recall"],
        "quantize_keys_ms": main_res["quantize_ms"],
        "extra": extra,
    }
    print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
