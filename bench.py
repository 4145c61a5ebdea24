#!/usr/bin/env python
"""Benchmark of the paged-KV hot path on GB300.

One step = one pass of the whole hot path over one decode batch of the chosen
workload, through the C ABI (libpkv.so):
  1. pkv_compute_slot_mapping  -- slot of every sequence's new token (position ctx-1)
  2. pkv_store_kvcache         -- scatter the new K/V rows into the paged caches
  3. pkv_paged_attention_decode -- one query per sequence over its whole paged
                                  context (main pass + split-K combine)
  4. pkv_unpack_block_paged x2 -- the batch's cache read as a CSR block-paged
                                  snapshot, unpacked for the key and value roles

`value` is the step's algorithmic HBM bytes divided by the device time of
the step (GB/s, inputs resident in HBM).  `e2e` is the same metric when
every step also copies its per-step inputs from pinned host memory and reads
the attention output back.  `roofline` is the decode-attention call
(the dominant kernel), timed back to back as a decode loop issues it, against
the measured HBM copy bandwidth; its per-call latency figure (one call between
two events after an L2 eviction) is reported beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]
For N > 1 launch under torch.distributed.run: every rank runs its own
replica of the workload (independent sequences, no collective on the data
path); the timed region is bracketed by barriers and the max over ranks is used.
"""
from __future__ import annotations

import argparse
import ctypes
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import pkv_workloads as wl  # noqa: E402

METRIC = "paged decode-attention KV GB/s and % of GB300 HBM roofline; decode tokens/s"
DEFAULT_CONFIG = "llama2-7b-layer-fp16"
DECODE_CONFIGS = ["llama2-7b-layer-fp16", "qwen3-0.6b-gqa-bf16", "long-gqa-8k-bf16", "long-gqa-32k-bf16",
                  "qwen3-0.6b-gqa-bf16-b1024"]
CSR_CONFIGS = ["csr-prefix-bf16"]
DTYPE_NAME = {torch.float16: "f16", torch.bfloat16: "bf16", torch.float32: "f32"}
HBM_FALLBACK_GBS = 6800.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=DECODE_CONFIGS + CSR_CONFIGS, default=DEFAULT_CONFIG)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-budget-s", type=float, default=12.0,
                    help="wall-clock budget of the oracle CPU-baseline sample")
    ap.add_argument("--window-s", type=float, default=1.0,
                    help="device time of every throughput window (profiler runs pass 0: one graph replay each)")
    ap.add_argument("--no-sweep", action="store_true",
                    help="measure only --config (skip the other decode workloads of the per-workload block)")
    ap.add_argument("--skip-cpu-baseline", action="store_true",
                    help="omit the oracle timing (for profiler runs)")
    ap.add_argument("--profile-calls", choices=["decode", "fp8", "int8", "prefill", "unpack", "store"], default=None,
                    help="profiler driver: run --steps calls of one kernel on the workload back to back, eagerly, "
                         "and exit without timing (decode attention over 16-bit, E4M3 or int8 caches; the chunked "
                         "prefill; the unpack of the batch's CSR snapshot (key role); the store of every context "
                         "token's K/V row, as after a prefill)")
    return ap.parse_args(argv)


# ----------------------------------------------------------------------------- distributed
def dist_init(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def reduce_max(x: float, world: int, device) -> float:
    """Max of a host scalar over ranks (timing only; nothing on the data path)."""
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ----------------------------------------------------------------------------- accounting
def step_bytes(cfg: wl.DecodeConfig, ctx: torch.Tensor, nnz: int) -> dict:
    """Algorithmic HBM bytes of one step, per kernel (what the computation must
    move at minimum; split-K partials are implementation overhead, not counted)."""
    es = torch.tensor([], dtype=cfg.dtype).element_size()
    B = int(ctx.numel())
    T = int(ctx.to(torch.int64).sum())
    row = cfg.num_kv_heads * cfg.head_dim * es
    q_bytes = B * cfg.num_q_heads * cfg.head_dim * es
    return {
        "slot_mapping": B * (4 * 4 + 4),                     # starts, ends, cu_new, table entry; slot out
        "store_kvcache": B * 4 + 2 * B * row * 2,            # slots; K and V rows read and written
        "paged_attention_decode": T * 2 * row + 2 * q_bytes + nnz * 4 + B * 4,  # KV once, q, out, tables
        "unpack_k": 2 * T * row + nnz * 4 + (B + 1) * 12,    # rows read and written, index buffers
        "unpack_v": 2 * T * row + nnz * 4 + (B + 1) * 12,
    }


def code8_attention_bytes(cfg: wl.DecodeConfig, ctx: torch.Tensor, nnz: int) -> int:
    """Algorithmic bytes of decode attention over 8-bit (E4M3 or int8) caches:
    one byte per K/V element, a K and a V scale per (block, head), q, out and
    the tables."""
    es = torch.tensor([], dtype=cfg.dtype).element_size()
    B, T = int(ctx.numel()), int(ctx.to(torch.int64).sum())
    return (T * 2 * cfg.num_kv_heads * cfg.head_dim + 2 * B * cfg.num_q_heads * cfg.head_dim * es + nnz * 4 + B * 4
            + nnz * cfg.num_kv_heads * 8)


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return HBM_FALLBACK_GBS, "fallback"


def measured_bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def profiled_traffic(kernel_key: str, units: float):
    """DRAM bytes per launch from a committed ncu summary, scaled to `units`,
    or None when the summary was taken on a different kernel source."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel_key]
        h = hashlib.sha256()  # every source file of the kernel, in the listed order
        for src in rec["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != rec["sources_sha256"]:
            return None
        return rec["dram_bytes_per_unit"] * units
    except (OSError, KeyError, ValueError, TypeError):
        return None


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        self.thread = None
        self.device_index = device_index

    def _gpu_selector(self):
        try:
            u = str(torch.cuda.get_device_properties(self.device_index).uuid)
            return u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            return vis.split(",")[self.device_index] if vis else str(self.device_index)

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
               "-lms", "100", "-i", self._gpu_selector()]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        used = inside if inside else self.samples
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"],
                    "samples_in_timed_region": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [v for v in (num(p[0]) for _, p in used) if v is not None]
        smax = [v for v in (num(p[1]) for _, p in used) if v is not None]
        reasons = set()
        for _, p in used:
            for name, val in zip(["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"],
                                 p[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        power = [v for v in (num(p[2]) for _, p in used) if v is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples_in_timed_region": len(inside),
                "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------------------- the step
def packed_inputs(tensors):
    """The per-step input tensors of one input set laid out in one device
    buffer (256-byte aligned offsets) and one pinned host buffer of the same
    layout, so that a step's inputs cross the link in a single copy.  Returns
    (device views with the tensors' data, host buffer, device buffer)."""
    offs, total = [], 0
    for t in tensors:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    dev = torch.zeros(max(total, 256), dtype=torch.uint8, device=tensors[0].device)
    views = []
    for t, o in zip(tensors, offs):
        v = dev[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
        v.copy_(t)
        views.append(v)
    host = dev.cpu().pin_memory()
    return views, host, dev


class DecodeStep:
    """Device buffers and C-ABI argument tuples of one hot-path step.

    `copies` > 1 keeps that many copies of the caches (same block tables, same
    values) so that a timed loop can rotate over them: consecutive calls then
    never find the previous call's K/V in L2 when one call reads less than the
    L2 holds a few times over."""

    def __init__(self, pkv, cfg: wl.DecodeConfig, seed: int, device):
        self.pkv, self.cfg, self.device = pkv, cfg, device
        self.batch = b = wl.decode_batch(cfg, seed=seed, device=device)
        self.snap = wl.decode_batch_snapshot(b)
        B, bs = cfg.batch, cfg.block_size
        self.B = B
        self.nb = b.extra["num_blocks"]
        self.slots = torch.empty(B, dtype=torch.int32, device=device)
        self.out = torch.empty_like(b.q)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        H, d = cfg.num_kv_heads, cfg.head_dim
        self.unpacked_k = None  # allocated on the first step that unpacks
        self.ws_bytes = pkv.pkv_paged_attention_decode_workspace_size(B, cfg.num_q_heads, H, d, bs,
                                                                      b.max_context_len, cfg.dtype)
        self.workspace = torch.zeros(max(self.ws_bytes, 256), dtype=torch.uint8, device=device)
        self.plan = pkv.pkv_paged_attention_decode_plan(B, cfg.num_q_heads, H, d, bs, b.max_context_len, cfg.dtype)
        self.dt = pkv._DTYPE[cfg.dtype]
        self.ctx_cpu = b.context_lens.cpu()
        self.bytes = step_bytes(cfg, self.ctx_cpu, self.snap.nnz)
        self.caches = [(b.k_cache, b.v_cache)]
        self.codes = []  # per copy: (k codes, v codes, k scales, v scales) of the 8-bit format self.code_fmt
        self.code_fmt = None
        # attention: main kernel + combine (always in the work-balanced schedule,
        # partition 0; with fixed partitions only when there is more than one)
        combine = self.plan[2] and self.plan[0] == 0 or self.plan[1] > 1
        self.attention_launches = 2 if combine else 1
        self.launches_per_step = 1 + 1 + self.attention_launches + 2

    def set_copies(self, n: int):
        """Keep n copies of the caches (the first is the batch's own)."""
        b = self.batch
        self.caches = self.caches[:n]
        while len(self.caches) < n:
            self.caches.append((b.k_cache.clone(), b.v_cache.clone()))

    def _unpack_buffers(self):
        if self.unpacked_k is None:
            c = self.cfg
            self.unpacked_k = torch.empty(self.snap.total_tokens, c.num_kv_heads, c.head_dim, dtype=c.dtype,
                                          device=self.device)
            self.unpacked_v = torch.empty_like(self.unpacked_k)

    def input_sets(self):
        """Two sets of the step's per-step device inputs (and outputs), so a
        pipelined loop can copy step i+1's inputs while step i runs.  Each set
        packs q, the new K/V rows, the tables, lengths, slot-mapping spans and
        CSR index buffers into one buffer (packed_inputs); the caches are
        shared."""
        if not hasattr(self, "_sets"):
            from dataclasses import replace

            b, s = self.batch, self.snap
            self._sets, self._packed = [], []
            for k in range(2):
                (q, nk, nv, bt, cl, st, en, cu), host, dev = packed_inputs(
                    [b.q, b.new_key, b.new_value, b.block_tables, b.context_lens, b.starts, b.ends, b.cu_new])
                bk = replace(b, q=q, new_key=nk, new_value=nv, block_tables=bt, context_lens=cl, starts=st, ends=en,
                             cu_new=cu)
                self._sets.append((bk, s, self.out if k == 0 else torch.empty_like(self.out)))
                self._packed.append((host, dev))
        return self._sets

    def run_set(self, stream_ptr, k: int, unpack: bool = True):
        """Enqueue one step on input set k (see input_sets)."""
        keep = (self.batch, self.snap, self.out)
        self.batch, self.snap, self.out = self.input_sets()[k]
        try:
            self.run(stream_ptr, unpack=unpack)
        finally:
            self.batch, self.snap, self.out = keep

    def run(self, stream_ptr, events=None, unpack: bool = True):
        """Enqueue one step; events (6 per step) bracket the kernels if given.
        unpack=False stops after the attention (a decode step)."""
        L, b, c, p = self.pkv._lib, self.batch, self.cfg, lambda t: t.data_ptr()
        rec = (lambda i: events[i].record()) if events is not None else (lambda i: None)
        ok = 0
        rec(0)
        ok |= L.pkv_compute_slot_mapping(p(b.block_tables), b.block_tables.shape[1], p(b.starts), p(b.ends),
                                         p(b.cu_new), self.B, c.block_size, self.nb, p(self.slots), self.B,
                                         p(self.err), stream_ptr)
        rec(1)
        ok |= L.pkv_store_kvcache(p(b.new_key), p(b.new_value), p(b.k_cache), p(b.v_cache), p(self.slots), self.B,
                                  c.num_kv_heads, c.head_dim, self.nb * c.block_size, self.dt, p(self.err),
                                  stream_ptr)
        rec(2)
        ok |= self.attention(stream_ptr)
        rec(3)
        if unpack:
            self._unpack_buffers()
            s = self.snap
            for pool, dst in ((b.k_cache, self.unpacked_k), (b.v_cache, self.unpacked_v)):
                ok |= L.pkv_unpack_block_paged(p(dst), p(pool), p(s.block_table), p(s.seq_ptr), self.pkv.PKV_U32,
                                               p(s.token_ptr), self.B, s.nnz, c.block_size, self.nb, c.num_kv_heads,
                                               c.head_dim, s.total_tokens, self.dt, p(self.err), stream_ptr)
                rec(4 if dst is self.unpacked_k else 5)
        if ok != 0:
            raise RuntimeError("pkv call failed: " + L.pkv_last_error_string().decode())

    def attention(self, stream_ptr, k: int = 0) -> int:
        """Enqueue the decode-attention call alone on cache copy k; returns its status."""
        L, b, c, p = self.pkv._lib, self.batch, self.cfg, lambda t: t.data_ptr()
        kc, vc = self.caches[k] if k else (b.k_cache, b.v_cache)
        return L.pkv_paged_attention_decode(p(self.out), p(b.q), p(kc), p(vc), p(b.block_tables),
                                            b.block_tables.shape[1], p(b.context_lens), self.B, c.num_q_heads,
                                            c.num_kv_heads, c.head_dim, c.block_size, self.nb, b.max_context_len,
                                            b.scale, self.dt, p(self.workspace), self.workspace.numel(),
                                            p(self.err), stream_ptr)

    def make_codes(self, fmt: str):
        """8-bit copies (fmt "fp8" = E4M3 or "int8"; per-(block, head) scales)
        of every cache copy, for the 8-bit passes; one format is held at a time."""
        self.codes = []
        quant = getattr(self.pkv, "pkv_quantize_kvcache_" + fmt)
        kq, ks = quant(self.caches[0][0])
        vq, vs = quant(self.caches[0][1])
        self.codes.append((kq, vq, ks, vs))
        for _ in range(1, len(self.caches)):
            self.codes.append((kq.clone(), vq.clone(), ks, vs))
        self.code_fmt = fmt

    def drop_codes(self):
        self.codes, self.code_fmt = [], None

    def code8_attention(self, stream_ptr, k: int = 0) -> int:
        """Enqueue the decode-attention call over the 8-bit caches of make_codes (copy k)."""
        L, b, c, p = self.pkv._lib, self.batch, self.cfg, lambda t: t.data_ptr()
        kq, vq, ks, vs = self.codes[k]
        fn = getattr(L, "pkv_paged_attention_decode_" + self.code_fmt)
        return fn(p(self.out), p(b.q), p(kq), p(vq), p(ks), p(vs), p(b.block_tables),
                  b.block_tables.shape[1], p(b.context_lens), self.B, c.num_q_heads, c.num_kv_heads, c.head_dim,
                  c.block_size, self.nb, b.max_context_len, b.scale, self.dt, p(self.workspace),
                  self.workspace.numel(), p(self.err), stream_ptr)

    def fused_step(self, stream_ptr, k: int = 0) -> int:
        """Enqueue the fused decode step (append the new K/V rows, then attend) on cache copy k."""
        L, b, c, p = self.pkv._lib, self.batch, self.cfg, lambda t: t.data_ptr()
        kc, vc = self.caches[k] if k else (b.k_cache, b.v_cache)
        return L.pkv_paged_attention_decode_append(p(self.out), p(b.q), p(b.new_key), p(b.new_value), p(kc), p(vc),
                                                   p(b.block_tables), b.block_tables.shape[1],
                                                   p(b.context_lens), self.B, c.num_q_heads, c.num_kv_heads,
                                                   c.head_dim, c.block_size, self.nb, b.max_context_len, b.scale,
                                                   self.dt, p(self.workspace), self.workspace.numel(), p(self.err),
                                                   stream_ptr)

    def separate_step(self, stream_ptr, k: int = 0) -> int:
        """Enqueue the same decode step as three calls: slot mapping, store, attention (cache copy k)."""
        L, b, c, p = self.pkv._lib, self.batch, self.cfg, lambda t: t.data_ptr()
        kc, vc = self.caches[k] if k else (b.k_cache, b.v_cache)
        st = L.pkv_compute_slot_mapping(p(b.block_tables), b.block_tables.shape[1], p(b.starts), p(b.ends),
                                        p(b.cu_new), self.B, c.block_size, self.nb, p(self.slots), self.B,
                                        p(self.err), stream_ptr)
        st |= L.pkv_store_kvcache(p(b.new_key), p(b.new_value), p(kc), p(vc), p(self.slots), self.B,
                                  c.num_kv_heads, c.head_dim, self.nb * c.block_size, self.dt, p(self.err),
                                  stream_ptr)
        return st | self.attention(stream_ptr, k)

    # per-step host inputs for the end-to-end measurement
    def host_inputs(self, k: int = 0):
        """(pinned host buffer, device buffer) pairs of input set k: one pair."""
        self.input_sets()
        return [self._packed[k]]


STEPS_PER_GRAPH = 10
MIN_WINDOW_S = 1.0      # device time of every throughput window (clock samples every 100 ms fall inside)
GRAPH_TARGET_MS = 2.0   # calls per graph: about this much device time, so graph boundaries are rare
COLD_CALLS = 20         # per-call (cold) timings per workload


def capture_step_graph(step: DecodeStep, n_steps: int):
    """CUDA graph of n_steps hot-path steps (kernels chained by programmatic
    dependent launch)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ptr = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        for _ in range(n_steps):
            step.run(ptr)
    return g


def capture_pipelined_io_graph(step, n_steps: int, io, unpack: bool = True):
    """CUDA graph of n_steps steps as a decode loop with host inputs runs them:
    step i reads input set i % 2, whose host->device copies run on a second
    stream as soon as step i - 2 is done with that set (overlapping step
    i - 1), and the device->host read of step i's output runs on that stream
    after step i while step i + 1 computes.  io = (per-set host/device input
    pairs, per-set pinned output, pinned error flag)."""
    pairs, out_host, err_host = io
    sets = step.input_sets()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(device=step.device)
    with torch.cuda.graph(g):
        comp = torch.cuda.current_stream()
        ptr = ctypes.c_void_p(comp.cuda_stream)
        ready = [torch.cuda.Event() for _ in range(n_steps)]
        done = [torch.cuda.Event() for _ in range(n_steps)]
        drained = [torch.cuda.Event() for _ in range(n_steps)]
        side.wait_stream(comp)
        for i in range(n_steps):
            k = i % 2
            with torch.cuda.stream(side):
                if i >= 2:
                    side.wait_event(done[i - 2])  # set k's inputs are no longer read
                for h, d in pairs[k]:
                    d.copy_(h, non_blocking=True)
                ready[i].record(side)
            comp.wait_event(ready[i])
            if i >= 2:
                comp.wait_event(drained[i - 2])  # output k has been read back
            if unpack:
                step.run_set(ptr, k)
            else:
                step.run_set(ptr, k, unpack=False)
            done[i].record(comp)
            with torch.cuda.stream(side):
                side.wait_event(done[i])
                out_host[k].copy_(sets[k][2], non_blocking=True)
                err_host.copy_(step.err, non_blocking=True)
                drained[i].record(side)
        comp.wait_stream(side)
    return g


def time_graphs(step, steps: int, world: int, io=None):
    """Replays graphs of STEPS_PER_GRAPH steps (and single steps for the
    remainder) so that exactly `steps` steps run between the two events; with
    io, the graphs are the pipelined end-to-end loop."""
    cap = (lambda n: capture_pipelined_io_graph(step, n, io)) if io is not None else \
        (lambda n: capture_step_graph(step, n))
    big = cap(STEPS_PER_GRAPH) if steps >= STEPS_PER_GRAPH else None
    one = cap(1)
    for _ in range(3):
        one.replay()
    if big is not None:
        big.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    e0.record()
    for _ in range(steps // STEPS_PER_GRAPH if big is not None else 0):
        big.replay()
    for _ in range(steps % STEPS_PER_GRAPH if big is not None else steps):
        one.replay()
    e1.record()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(world)
    return e0.elapsed_time(e1), (t_wall0, t_wall1)


def replay_window(g, units_per_replay: int, world: int, min_s: float | None = None, min_units: int = 0):
    """Replays graph g back to back until at least min_s seconds of device time
    (and min_units units) have run between two CUDA events (min_s defaults to
    MIN_WINDOW_S).  Returns (ms per unit, units timed, (wall start, wall end))."""
    min_s = MIN_WINDOW_S if min_s is None else min_s
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    est = max(e0.elapsed_time(e1), 1e-3)
    n = max(1, math.ceil(min_s * 1e3 / est), math.ceil(min_units / units_per_replay))
    barrier(world)
    torch.cuda.synchronize()
    tw0 = time.time()
    e0.record()
    for _ in range(n):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    tw1 = time.time()
    barrier(world)
    return e0.elapsed_time(e1) / (n * units_per_replay), n * units_per_replay, (tw0, tw1)


def capture_calls(step, what, n_calls: int, ncopies: int = 1):
    """CUDA graph of n_calls calls of what(stream_ptr, copy), copy = i % ncopies
    (launches chained by programmatic dependent launch)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ptr = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        for i in range(n_calls):
            if what(ptr, i % ncopies) != 0:
                raise RuntimeError("pkv call failed: " + step.pkv._lib.pkv_last_error_string().decode())
    return g


def calls_per_graph(est_ms: float, ncopies: int) -> int:
    """About GRAPH_TARGET_MS of calls per graph (8 to 64), a multiple of ncopies."""
    n = min(64, max(8, math.ceil(GRAPH_TARGET_MS / max(est_ms, 1e-3))))
    return (n + ncopies - 1) // ncopies * ncopies


def time_sustained(step, what, world: int, est_ms: float, ncopies: int = 1, min_s: float | None = None,
                   min_calls: int = 0):
    """Calls of `what` back to back, as a decode loop issues them, rotating
    over ncopies cache copies, for at least min_s seconds of device time.
    Returns (ms per call, calls timed, calls per graph, wall window)."""
    per = calls_per_graph(est_ms, ncopies)
    g = capture_calls(step, what, per, ncopies)
    ms, calls, win = replay_window(g, per, world, min_s, min_calls)
    return ms, calls, per, win


_EVICT = {}


def evict_buffer(device):
    """A 512 MB buffer whose read evicts the L2 (and writes back its dirty lines)."""
    if device not in _EVICT:
        _EVICT[device] = (torch.ones(L2_EVICT_BYTES // 4, dtype=torch.float32, device=device),
                          torch.empty((), dtype=torch.float32, device=device))
    return _EVICT[device]


def time_cold_calls(step, what, n: int, world: int, stream):
    """One call at a time between two CUDA events on the launching stream,
    each after a 512 MB read (outside the events) that evicts the L2: launch
    latency and a cold L2 included.  Returns (median ms, mean ms)."""
    evict, sink = evict_buffer(step.device)
    ptr = ctypes.c_void_p(stream.cuda_stream)
    with torch.cuda.stream(stream):
        for _ in range(2):
            what(ptr, 0)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        torch.cuda.synchronize()
        barrier(world)
        for a, b in evs:
            torch.sum(evict, dim=0, out=sink)
            a.record()
            if what(ptr, 0) != 0:
                raise RuntimeError("pkv call failed: " + step.pkv._lib.pkv_last_error_string().decode())
            b.record()
        torch.cuda.synchronize()
        barrier(world)
    t = [a.elapsed_time(b) for a, b in evs]
    return statistics.median(t), statistics.fmean(t)


L2_EVICT_BYTES = 512 << 20  # > 4x the 129 MB L2


def l2_bytes(device) -> int:
    try:
        return int(torch.cuda.get_device_properties(device).L2_cache_size) or 129 * 10 ** 6
    except Exception:
        return 129 * 10 ** 6


def time_kernels(step: DecodeStep, steps: int, world: int, stream):
    """Per-kernel pass: eager launches with CUDA events between the kernels on
    the launching stream.  Before every step (outside the events) a 512 MB
    buffer is read, which evicts the L2 and writes back the previous step's
    dirty lines, so no kernel is charged for another kernel's deferred writes.
    The events cut the launch chaining, so these per-kernel times are slightly
    pessimistic."""
    ptr = ctypes.c_void_p(stream.cuda_stream)
    evict, sink = evict_buffer(step.device)
    with torch.cuda.stream(stream):
        for _ in range(3):
            step.run(ptr)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
        torch.cuda.synchronize()
        barrier(world)
        for i in range(steps):
            torch.sum(evict, dim=0, out=sink)
            step.run(ptr, evs[i])
        torch.cuda.synchronize()
        barrier(world)
    names = ["slot_mapping", "store_kvcache", "paged_attention_decode", "unpack_k", "unpack_v"]
    return {n: statistics.fmean(e[k].elapsed_time(e[k + 1]) for e in evs) for k, n in enumerate(names)}


def time_host_allocator(pkv, step: DecodeStep, steps: int = 200):
    """Host block allocator on the workload's pool: the batch's sequences are
    admitted with their context lengths, then every step appends one token to
    each (a new block whenever a length becomes 1 mod block_size).  Returns
    microseconds per decode step of bookkeeping, or None if the pool is too
    small for the extra tokens."""
    cfg = step.cfg
    a = pkv.pkv_allocator_create(step.nb, cfg.block_size)
    for i, n in enumerate(step.ctx_cpu.tolist()):
        pkv.pkv_allocator_add_sequence(a, i, n)
    if pkv.pkv_allocator_stats(a)["free"] < step.B * (steps // cfg.block_size + 1):
        return None
    t0 = time.perf_counter()
    for _ in range(steps):
        for i in range(step.B):
            pkv.pkv_allocator_append(a, i)
    dt = time.perf_counter() - t0
    assert pkv.pkv_allocator_check(a) == 0
    return dt / steps * 1e6


PREFILL_NEW_TOKENS = 512


def prefill_call(step: DecodeStep):
    """Chunked prefill on the workload's own cache: every sequence's last
    min(ctx, 512) positions are taken as the new tokens of a prefill chunk
    (fresh random queries) and attend causally over their whole context.
    Returns (enqueue function (stream_ptr, copy), algorithmic FLOPs per call,
    queries): 2 d flops for q.k and 2 d for p.v per (query, key) pair and
    query head."""
    pkv, b, c = step.pkv, step.batch, step.cfg
    ctx = step.ctx_cpu.to(torch.int64)
    ns = ctx.clamp(max=PREFILL_NEW_TOKENS)
    starts = (ctx - ns).to(torch.int32)
    cu = torch.zeros(step.B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(ns, 0).to(torch.int32)
    nq = int(cu[-1])
    pairs = int(sum(int(n) * int(s) + int(n) * (int(n) + 1) // 2 for s, n in zip(starts, ns)))
    flops = pairs * 4 * c.head_dim * c.num_q_heads
    g = torch.Generator(device=step.device).manual_seed(11)
    q = torch.randn(nq, c.num_q_heads, c.head_dim, generator=g, device=step.device).to(c.dtype)
    out = torch.empty_like(q)
    st, cud = starts.to(step.device), cu.to(step.device)
    L, p = pkv._lib, lambda t: t.data_ptr()
    mq = int(ns.max())

    def call(ptr, k=0):
        return L.pkv_paged_attention_prefill(p(out), p(q), p(b.k_cache), p(b.v_cache), p(b.block_tables),
                                             b.block_tables.shape[1], p(st), p(cud), step.B, mq, c.num_q_heads,
                                             c.num_kv_heads, c.head_dim, c.block_size, step.nb, b.scale, step.dt,
                                             p(step.err), ptr)

    step.prefill_buffers = (q, out, st, cud)  # kept alive with the step
    return call, flops, nq


def e2e_io(step):
    """Pinned host buffers of the end-to-end pass, per input set."""
    pairs = [step.host_inputs(0), step.host_inputs(1)]
    out_host = [torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory() for _ in range(2)]
    err_host = torch.empty(1, dtype=torch.int32).pin_memory()
    h2d = sum(h.numel() * h.element_size() for h, _ in pairs[0])
    d2h = out_host[0].numel() * out_host[0].element_size() + 4
    return (pairs, out_host, err_host), h2d, d2h


# ----------------------------------------------------------------------------- oracle sample
def oracle_sample_inputs(batch: wl.DecodeBatch, seqs):
    """The chosen sequences with only the blocks they use, on the CPU (block
    ids renumbered into a compact pool)."""
    bs = batch.cfg.block_size
    ctx = batch.context_lens.cpu()[seqs]
    tables = batch.block_tables.cpu()[seqs]
    nblk = [(int(c) + bs - 1) // bs for c in ctx]
    used = torch.cat([tables[i, :n] for i, n in enumerate(nblk)]).to(torch.int64)
    remap = {int(x): i for i, x in enumerate(used.tolist())}
    new_tables = torch.full((len(seqs), max(nblk)), -1, dtype=torch.int32)
    for i, n in enumerate(nblk):
        new_tables[i, :n] = torch.tensor([remap[int(x)] for x in tables[i, :n]], dtype=torch.int32)
    kc = batch.k_cache[used.to(batch.k_cache.device)].cpu()
    vc = batch.v_cache[used.to(batch.v_cache.device)].cpu()
    return dict(q=batch.q.cpu()[seqs], kc=kc, vc=vc, tables=new_tables, ctx=ctx, nnz=len(used))


def oracle_attention(orc, s, scale):
    """The decode attention of one sample, computed by the oracle."""
    orc.paged_attention_decode(s["q"], s["kc"], s["vc"], s["tables"], s["ctx"], scale)


def cpu_sample_run(batch, budget_s: float, start_seq: int = 0, max_seqs: int | None = None):
    """Decode attention by the oracle over sequences start_seq, start_seq+1, ...
    (one at a time, inputs gathered outside the clock) until the budget is
    spent; returns (KV GB/s, seconds, number of sequences, bytes), bytes being
    the attention's algorithmic bytes of those sequences."""
    import oracle as orc

    orc.build()
    cfg, B = batch.cfg, batch.cfg.batch
    done, t_total, nbytes = 0, 0.0, 0
    while t_total < budget_s and (max_seqs is None or done < max_seqs) and done < B:
        seq = [(start_seq + done) % B]
        s = oracle_sample_inputs(batch, seq)
        t0 = time.perf_counter()
        oracle_attention(orc, s, batch.scale)
        t_total += time.perf_counter() - t0
        nbytes += step_bytes(cfg, s["ctx"], s["nnz"])["paged_attention_decode"]
        done += 1
    return nbytes / t_total / 1e9, t_total, done, nbytes


def cpu_all_cores_run(batch, max_seqs: int):
    """The same oracle attention on the first max_seqs sequences, one sequence
    per task on a pool of host threads (the C oracle runs outside the GIL);
    inputs are prepared before the clock starts.  Returns (GB/s, seconds,
    sequences, bytes, threads)."""
    import oracle as orc
    from concurrent.futures import ThreadPoolExecutor

    orc.build()
    cfg = batch.cfg
    n = min(max_seqs, cfg.batch)
    samples = [oracle_sample_inputs(batch, [i]) for i in range(n)]
    threads = max(1, min(len(os.sched_getaffinity(0)), n))
    with ThreadPoolExecutor(max_workers=threads) as pool:
        t0 = time.perf_counter()
        list(pool.map(lambda smp: oracle_attention(orc, smp, batch.scale), samples))
        secs = time.perf_counter() - t0
    nbytes = sum(step_bytes(cfg, smp["ctx"], smp["nnz"])["paged_attention_decode"] for smp in samples)
    return nbytes / secs / 1e9, secs, n, nbytes, threads


# ----------------------------------------------------------------------------- the workload description
def workload_config(cfg: wl.DecodeConfig, ctx: torch.Tensor, world: int) -> dict:
    """The `config` object of a decode workload: the same dict on both arms."""
    es = torch.tensor([], dtype=cfg.dtype).element_size()
    tokens = int(ctx.to(torch.int64).sum())
    kv = tokens * 2 * cfg.num_kv_heads * cfg.head_dim * es
    return {
        "workload": cfg.name, "description": cfg.description, "batch": cfg.batch,
        "num_q_heads": cfg.num_q_heads, "num_kv_heads": cfg.num_kv_heads, "head_dim": cfg.head_dim,
        "block_size": cfg.block_size, "context_tokens": tokens, "max_context_len": int(ctx.max()),
        "kv_bytes_per_call": kv,
        "l2": f"{kv / 1e9:.2f} GB of K/V per decode-attention call vs the 129 MB L2: no flush; workloads under "
              "4x L2 rotate over cache copies",
        "parallelism": f"replicas x{world} (independent sequences per rank, no data-path collective)",
    }


DEFAULT_SWEEP = ["llama2-7b-layer-fp16", "qwen3-0.6b-gqa-bf16", "long-gqa-8k-bf16", "long-gqa-32k-bf16",
                 "qwen3-0.6b-gqa-bf16-b1024"]


def _clk(summary: dict) -> dict:
    return {k: summary.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples_in_timed_region", "power_w_max")}


def measure_decode_workload(pkv, step: DecodeStep, world: int, device, stream, sampler) -> dict:
    """Decode attention on one workload: cold per-call latency, sustained
    calls (rotating over cache copies when a call reads under 4x L2), the
    fused decode step and the 8-bit caches, each sustained window at least
    MIN_WINDOW_S of device time."""
    cfg = step.cfg
    peak, _ = measured_hbm_peak()
    l2 = l2_bytes(device)
    kv_alg = step.bytes["paged_attention_decode"]
    ncopies = 1 if kv_alg >= 4 * l2 else max(4, math.ceil(4 * l2 / kv_alg))
    step.set_copies(ncopies)
    rmax = lambda x: reduce_max(x, world, device)  # noqa: E731
    rsum = lambda x: reduce_sum(x, world, device)  # noqa: E731
    all_bytes = rsum(kv_alg)
    B_all = rsum(cfg.batch)

    def gbs(nbytes, ms):
        return nbytes / (ms * 1e-3) / 1e9

    res = {"workload": cfg.name, "batch": cfg.batch, "context_tokens": int(step.ctx_cpu.to(torch.int64).sum()),
           "attention_bytes_per_call": kv_alg, "cache_copies": ncopies,
           "plan": {"partition_tokens": step.plan[0], "partitions_or_ctas": step.plan[1],
                    "tensor_core_path": step.plan[2],
                    "schedule": "work-balanced" if step.plan[2] and step.plan[0] == 0 else "fixed partitions"}}
    cold_med, cold_mean = time_cold_calls(step, step.attention, COLD_CALLS, world, stream)
    cold_med, cold_mean = rmax(cold_med), rmax(cold_mean)
    ms, calls, per, (t0, t1) = time_sustained(step, step.attention, world, cold_med, ncopies)
    clk = sampler.summary(t0, t1)
    ms = rmax(ms)
    a = gbs(all_bytes, ms)
    c = gbs(all_bytes, cold_med)
    res["attention"] = {
        "sustained": {"us": round(ms * 1e3, 2), "gbs": round(a, 1), "frac": round(a / peak, 4),
                      "frac_of_8000_nominal": round(a / 8000.0, 4), "calls": calls, "calls_per_graph": per,
                      "clocks": _clk(clk)},
        "per_call": {"us": round(cold_med * 1e3, 2), "us_mean": round(cold_mean * 1e3, 2), "gbs": round(c, 1),
                     "frac": round(c / peak, 4), "frac_of_8000_nominal": round(c / 8000.0, 4),
                     "calls": COLD_CALLS},
        "tokens_per_s": round(B_all / (ms * 1e-3), 1)}
    fms, fcalls, _, (t0, t1) = time_sustained(step, step.fused_step, world, ms, ncopies)
    fms = rmax(fms)
    res["decode_step_fused"] = {"us": round(fms * 1e3, 2), "tokens_per_s": round(B_all / (fms * 1e-3), 1),
                                "kv_gbs": round(gbs(all_bytes, fms), 1), "calls": fcalls,
                                "clocks": _clk(sampler.summary(t0, t1))}
    c8_bytes = rsum(code8_attention_bytes(cfg, step.ctx_cpu, step.snap.nnz))
    for fmt in ("fp8", "int8"):
        step.make_codes(fmt)
        ptr = ctypes.c_void_p(stream.cuda_stream)
        with torch.cuda.stream(stream):
            st = step.code8_attention(ptr, 0)
        torch.cuda.synchronize()
        if st != 0:
            res[fmt] = {"unsupported": pkv._lib.pkv_last_error_string().decode()}
            step.drop_codes()
            continue
        c8_local = code8_attention_bytes(cfg, step.ctx_cpu, step.snap.nnz)
        n8 = 1 if c8_local >= 4 * l2 else max(4, math.ceil(4 * l2 / c8_local))
        m8, calls8, _, (t0, t1) = time_sustained(step, step.code8_attention, world, ms / 2, min(n8, len(step.codes)))
        m8 = rmax(m8)
        g8 = gbs(c8_bytes, m8)
        res[fmt] = {"us": round(m8 * 1e3, 2), "gbs": round(g8, 1), "frac": round(g8 / peak, 4),
                    "frac_of_8000_nominal": round(g8 / 8000.0, 4), "tokens_per_s": round(B_all / (m8 * 1e-3), 1),
                    "speedup_vs_16bit": round(ms / m8, 3), "calls": calls8,
                    "clocks": _clk(sampler.summary(t0, t1))}
        step.drop_codes()
    step.set_copies(1)
    torch.cuda.synchronize()
    err = int(step.err.item())
    if err:
        raise RuntimeError(f"device error bits {err:#x} during the {cfg.name} passes")
    return res


# ----------------------------------------------------------------------------- arms
def run_reference(args, world, rank):
    """The oracle as it stands, on the host cores: decode attention of a
    bounded sample of the workload's sequences per step."""
    if rank != 0:
        return 0
    cfg = wl.CONFIGS[args.config]
    device = "cuda" if torch.cuda.is_available() else "cpu"
    batch = wl.decode_batch(cfg, seed=args.seed, device=device)
    seqs_per_step = 2
    for w in range(args.warmup):
        cpu_sample_run(batch, 1e9, start_seq=w * seqs_per_step, max_seqs=seqs_per_step)
    t, nbytes = 0.0, 0
    for i in range(args.steps):
        _, dt, _, nb = cpu_sample_run(batch, 1e9, start_seq=(args.warmup + i) * seqs_per_step,
                                      max_seqs=seqs_per_step)
        t += dt
        nbytes += nb
    value = nbytes / t / 1e9
    sample = (f"{seqs_per_step} sequences of the {cfg.name} batch per step, decode attention of each over its "
              "whole paged context; single-threaded C oracle in binary64")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_NAME[cfg.dtype],
        "data": "synthetic (seeded N(0,1) K/V/q, random non-contiguous block permutation)",
        "config": workload_config(cfg, batch.context_lens.cpu(), world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, world, rank, local):
    import pagedattention_decode_pkv_gb300 as pkv

    global MIN_WINDOW_S
    MIN_WINDOW_S = args.window_s

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    cfg = wl.CONFIGS[args.config]
    step = DecodeStep(pkv, cfg, seed=args.seed + rank, device=device)
    stream = torch.cuda.Stream(device)
    rmax = lambda x: reduce_max(x, world, device)  # noqa: E731
    rsum = lambda x: reduce_sum(x, world, device)  # noqa: E731

    # eager warm-up: first-use set-up of the library, then the graphs
    ptr = ctypes.c_void_p(stream.cuda_stream)
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step.run(ptr)
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    try:
        # 1. exactly `steps` hot-path steps (slot mapping, store, attention, unpack K and V)
        total_ms, (tw0, tw1) = time_graphs(step, args.steps, world)
        clocks_steps = sampler.summary(tw0, tw1)
        torch.cuda.synchronize()
        if int(step.err.item()):
            raise RuntimeError(f"device error bits {int(step.err.item()):#x} during the benchmark")
        # 2. the headline: decode-attention calls back to back for >= 1 s
        headline = measure_decode_workload(pkv, step, world, device, stream, sampler)
        # 3. the other decode workloads, the same passes
        sweep = {cfg.name: headline}
        if not args.no_sweep:
            for name in DEFAULT_SWEEP:
                if name == cfg.name:
                    continue
                other = DecodeStep(pkv, wl.CONFIGS[name], seed=args.seed + rank, device=device)
                with torch.cuda.stream(stream):
                    other.attention(ptr)
                torch.cuda.synchronize()
                sweep[name] = measure_decode_workload(pkv, other, world, device, stream, sampler)
                del other
                torch.cuda.empty_cache()
        # 4. per-kernel times of the headline step, the separate decode step,
        #    the prefill, the end-to-end decode loop
        per = time_kernels(step, max(args.steps, COLD_CALLS), world, stream)
        sep_ms, _, _, _ = time_sustained(step, step.separate_step, world, per["paged_attention_decode"])
        sep_ms = rmax(sep_ms)
        call, pre_flops, pre_q = prefill_call(step)
        pre_ms, pre_calls, _, (t0, t1) = time_sustained(step, call, world, 1.5)
        pre_clk = sampler.summary(t0, t1)
        pre_ms = rmax(pre_ms)
        io, h2d, d2h = e2e_io(step)
        g_e2e = capture_pipelined_io_graph(step, STEPS_PER_GRAPH, io, unpack=False)
        e2e_ms, e2e_steps, (t0, t1) = replay_window(g_e2e, STEPS_PER_GRAPH, world)
        e2e_clk = sampler.summary(t0, t1)
        e2e_ms = rmax(e2e_ms)
    finally:
        sampler.stop()
    torch.cuda.synchronize()
    if int(step.err.item()):
        raise RuntimeError(f"device error bits {int(step.err.item()):#x} during the benchmark")
    alloc_us = time_host_allocator(pkv, step)

    peak, peak_kind = measured_hbm_peak()
    bf16_peak, bf16_kind = measured_bf16_peak()
    attn_bytes = step.bytes["paged_attention_decode"]
    all_attn_bytes = rsum(attn_bytes)
    h_sus = headline["attention"]["sustained"]
    value = h_sus["gbs"]
    step_total_bytes = sum(step.bytes.values())
    total_ms_max = rmax(total_ms)
    step_gbs = rsum(step_total_bytes * args.steps) / (total_ms_max * 1e-3) / 1e9
    e2e_value = all_attn_bytes / (e2e_ms * 1e-3) / 1e9
    units = int(step.ctx_cpu.to(torch.int64).sum())  # tokens of context per launch
    traffic = profiled_traffic("paged_attention_decode", units)
    roof_calls = h_sus["calls"]

    cpu_baseline = None
    if world == 1 and not args.skip_cpu_baseline:
        gbs, secs, nseq, nbytes = cpu_sample_run(step.batch, args.cpu_budget_s)
        cpu_baseline = {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                        "sample": f"decode attention of the first {nseq} of {cfg.batch} sequences of the batch, one "
                                  f"sequence at a time ({nbytes / 1e9:.3f} GB of attention bytes in {secs:.1f} s), "
                                  "single-threaded C oracle in binary64"}
        mgbs, msecs, mseq, mbytes, threads = cpu_all_cores_run(step.batch, max(nseq, 1))
        cpu_baseline["all_cores"] = {
            "value": round(mgbs, 4), "unit": "GB/s", "cores": threads,
            "sample": f"the same {mseq} sequences ({mbytes / 1e9:.3f} GB in {msecs:.2f} s), one sequence per task "
                      f"on {threads} host threads"}

    if rank != 0:
        return 0
    kernel_us = {k: round(v * 1e3, 2) for k, v in per.items()}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": round(total_ms_max / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_NAME[cfg.dtype],
        "data": "synthetic (seeded N(0,1) K/V/q, random non-contiguous block permutation)",
        "config": workload_config(cfg, step.ctx_cpu, world),
        "plan": headline["plan"],
        "decode_tokens_per_s": headline["decode_step_fused"]["tokens_per_s"],
        "attention_tokens_per_s": headline["attention"]["tokens_per_s"],
        "step_gbs": round(step_gbs, 2),
        "step_bytes": step_total_bytes,
        "kernel_us": kernel_us,
        "kernel_gbs": {k: round(step.bytes[k] / (per[k] * 1e-3) / 1e9, 1) for k in per},
        "roofline": {"kernel": "pkv_paged_attention_decode (main pass + merge)", "bound": "hbm",
                     "achieved": value, "peak": peak, "unit": "GB/s", "frac": round(value / peak, 4),
                     "peak_kind": peak_kind, "frac_of_8000_nominal": round(value / 8000.0, 4),
                     "traffic": None if traffic is None else round(traffic),
                     "algorithmic_bytes_per_call": attn_bytes,
                     "us_per_call": h_sus["us"], "calls_timed": roof_calls,
                     "per_call_latency": headline["attention"]["per_call"]},
        "configs": sweep,
        "decode_step_separate_us": round(sep_ms * 1e3, 2),
        "prefill": {
            "what": f"pkv_paged_attention_prefill: each sequence's last min(ctx, {PREFILL_NEW_TOKENS}) positions as a "
                    "prefill chunk over its own paged context (causal), back to back in CUDA graphs",
            "queries": pre_q, "us_per_call": round(pre_ms * 1e3, 2), "calls": pre_calls,
            "clocks": _clk(pre_clk),
            "roofline": {"bound": "tensor", "achieved": round(pre_flops / (pre_ms * 1e-3) / 1e12, 2),
                         "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": round(pre_flops / (pre_ms * 1e-3) / 1e12 / bf16_peak, 4),
                         "peak_kind": bf16_kind, "flops_per_call": pre_flops}},
        "host_allocator_us_per_step": None if alloc_us is None else round(alloc_us, 1),
        "cpu_baseline": cpu_baseline,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps,
                "clocks": _clk(e2e_clk)},
        "gpu_launches": step.launches_per_step * args.steps + step.attention_launches * roof_calls,
        "timing": {
            "value": "decode-attention KV GB/s: algorithmic bytes of one pkv_paged_attention_decode call (K and V "
                     "once, q, out, tables) over the sustained time per call (main pass + merge); calls back to back "
                     f"in CUDA graphs (PDL-chained), graphs replayed for >= {MIN_WINDOW_S:.0f} s of device time "
                     "between two CUDA events; = roofline.achieved",
            "ms_per_step": f"exactly `steps` whole hot-path steps (slot mapping, store, attention, unpack K and V) in "
                           f"CUDA graphs of {STEPS_PER_GRAPH} steps between two CUDA events; step_gbs = their "
                           "algorithmic bytes over that time",
            "configs": "every decode workload: per_call = one call between two CUDA events after a 512 MB "
                       "L2-evicting read (median of 20, launch latency included); sustained = calls back to back for "
                       f">= {MIN_WINDOW_S:.0f} s, rotating over `cache_copies` copies of the caches when one call reads "
                       "under 4x L2; fp8/int8 = the same over E4M3/int8 caches (code bytes); decode_step_fused = "
                       "append + attention (pkv_paged_attention_decode_append), tokens/s = batch / its time",
            "kernel_us": "eager steps with CUDA events between the kernels on the launching stream; a 512 MB read "
                         "before each step (outside the events) evicts L2",
            "e2e": "decode steps (slot mapping, store, attention) as a pipelined loop runs them, for >= 1 s: every "
                   "step copies its inputs from pinned host memory in one copy (two device input sets, step i+1's "
                   "copy on a second stream overlaps step i) and reads its attention output and error flag back; "
                   "value = attention KV bytes per step over the step time",
            "gpu_launches": "kernels launched in the two timed regions value and ms_per_step come from"},
        "clocks": dict(h_sus["clocks"], steps_pass=_clk(clocks_steps)),
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- CSR prefix-shared workload
def csr_step_bytes(cfg: wl.CsrConfig, snap):
    """Per-kernel bytes of one CSR pass: unique (written rows plus every page
    row once: what HBM must move when shared pages are read once) and logical
    (every row a sequence names).  Returns (unique, logical, unique tokens)."""
    es = torch.tensor([], dtype=cfg.dtype).element_size()
    S, T, nnz = cfg.num_seqs, snap.total_tokens, int(snap.block_table.numel())
    row = cfg.num_heads * cfg.head_dim * es
    n_shared = int(cfg.num_seqs * cfg.shared_fraction)
    unique_tokens = T - max(n_shared - 1, 0) * cfg.prefix_tokens
    idx = nnz * 4 + (S + 1) * 12                        # block table, seq_ptr, token_ptr
    q_bytes = S * cfg.num_heads * cfg.head_dim * es
    tables = int(snap.block_tables_2d.numel()) * 4 + S * 4
    unique = {
        "unpack_k": T * row + unique_tokens * row + idx,
        "unpack_v": T * row + unique_tokens * row + idx,
        "paged_attention_decode": unique_tokens * 2 * row + 2 * q_bytes + tables,
    }
    logical = {
        "unpack_k": 2 * T * row + idx,
        "unpack_v": 2 * T * row + idx,
        "paged_attention_decode": T * 2 * row + 2 * q_bytes + tables,
    }
    return unique, logical, unique_tokens


class CsrStep:
    """One pass over a block-paged snapshot whose first half of the sequences
    alias the same prefix pages: unpack of K and of V into contiguous
    [total_tokens, H, d] buffers, and decode attention over the same pages
    through the padded 2-D table (Hq == Hkv == H).  Byte counts per kernel:
    logical (every row a sequence names) and unique (every page row once: what
    HBM must move when the shared pages are read once)."""

    def __init__(self, pkv, cfg: wl.CsrConfig, seed: int, device):
        self.pkv, self.cfg, self.device = pkv, cfg, device
        self.snap = s = wl.csr_snapshot(cfg, seed=seed, device=device)
        H, d = cfg.num_heads, cfg.head_dim
        es = torch.tensor([], dtype=cfg.dtype).element_size()
        self.dt = pkv._DTYPE[cfg.dtype]
        self.S, self.T, self.nnz = cfg.num_seqs, s.total_tokens, int(s.block_table.numel())
        self.num_pages = int(s.k_pool.shape[0])
        self.maxc = int(s.seq_lens.max())
        self.out_k = torch.empty(self.T, H, d, dtype=cfg.dtype, device=device)
        self.out_v = torch.empty_like(self.out_k)
        self.out = torch.empty_like(s.q)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        ws = pkv.pkv_paged_attention_decode_workspace_size(self.S, H, H, d, cfg.page_size, self.maxc, cfg.dtype)
        self.workspace = torch.zeros(max(ws, 256), dtype=torch.uint8, device=device)
        self.bytes, self.logical, self.unique_tokens = csr_step_bytes(cfg, s)

    def _unpack(self, stream_ptr, dst, pool, s) -> int:
        L, p, c = self.pkv._lib, (lambda t: t.data_ptr()), self.cfg
        return L.pkv_unpack_block_paged(p(dst), p(pool), p(s.block_table), p(s.seq_ptr), self.pkv.PKV_U32,
                                        p(s.token_ptr), self.S, self.nnz, c.page_size, self.num_pages, c.num_heads,
                                        c.head_dim, self.T, self.dt, p(self.err), stream_ptr)

    def attention(self, stream_ptr) -> int:
        L, p, c, s = self.pkv._lib, (lambda t: t.data_ptr()), self.cfg, self.snap
        return L.pkv_paged_attention_decode(p(self.out), p(s.q), p(s.k_pool), p(s.v_pool), p(s.block_tables_2d),
                                            s.block_tables_2d.shape[1], p(s.seq_lens), self.S, c.num_heads,
                                            c.num_heads, c.head_dim, c.page_size, self.num_pages, self.maxc,
                                            s.scale, self.dt, p(self.workspace), self.workspace.numel(),
                                            p(self.err), stream_ptr)

    def run(self, stream_ptr, events=None):
        """Enqueue one pass (unpack K, unpack V, attention); events (4) bracket the kernels if given."""
        rec = (lambda i: events[i].record()) if events is not None else (lambda i: None)
        s = self.snap
        rec(0)
        ok = self._unpack(stream_ptr, self.out_k, s.k_pool, s)
        rec(1)
        ok |= self._unpack(stream_ptr, self.out_v, s.v_pool, s)
        rec(2)
        ok |= self.attention(stream_ptr)
        rec(3)
        if ok != 0:
            raise RuntimeError("pkv call failed: " + self.pkv._lib.pkv_last_error_string().decode())

    # pipelined end-to-end loop: per-step inputs are q and the index buffers; the pools are resident
    def input_sets(self):
        """Two packed input sets (packed_inputs) for the pipelined loop."""
        if not hasattr(self, "_sets"):
            from dataclasses import replace

            s = self.snap
            self._sets, self._packed = [], []
            for k in range(2):
                (q, bt, sp, tp, sl, bt2), host, dev = packed_inputs(
                    [s.q, s.block_table, s.seq_ptr, s.token_ptr, s.seq_lens, s.block_tables_2d])
                sk = replace(s, q=q, block_table=bt, seq_ptr=sp, token_ptr=tp, seq_lens=sl, block_tables_2d=bt2)
                self._sets.append((sk, None, self.out if k == 0 else torch.empty_like(self.out)))
                self._packed.append((host, dev))
        return self._sets

    def run_set(self, stream_ptr, k: int):
        keep = (self.snap, self.out)
        self.snap, _, self.out = self.input_sets()[k]
        try:
            self.run(stream_ptr)
        finally:
            self.snap, self.out = keep

    def host_inputs(self, k: int = 0):
        self.input_sets()
        return [self._packed[k]]


def time_csr_kernels(step: CsrStep, steps: int, world: int, stream):
    """Per-call times of the three kernels: eager launches with events between
    them, a 512 MB L2-evicting read before every pass (outside the events)."""
    ptr = ctypes.c_void_p(stream.cuda_stream)
    evict = torch.ones(L2_EVICT_BYTES // 4, dtype=torch.float32, device=step.device)
    sink = torch.empty((), dtype=torch.float32, device=step.device)
    with torch.cuda.stream(stream):
        for _ in range(3):
            step.run(ptr)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        torch.cuda.synchronize()
        barrier(world)
        for i in range(steps):
            torch.sum(evict, dim=0, out=sink)
            step.run(ptr, evs[i])
        torch.cuda.synchronize()
        barrier(world)
    names = ["unpack_k", "unpack_v", "paged_attention_decode"]
    return {n: statistics.fmean(e[k].elapsed_time(e[k + 1]) for e in evs) for k, n in enumerate(names)}


def csr_oracle_run(s, step_bytes_total: int, max_seqs: int, budget_s: float):
    """The oracle on whole sequences of the snapshot, one at a time (each
    sequence's pages gathered into a compact pool first, outside the clock):
    unpack of K and V and decode attention.  Returns (GB/s, seconds,
    sequences, bytes), the bytes being the sequences' share of the pass's
    unique bytes (their tokens over all tokens)."""
    import oracle as orc

    orc.build()
    bt, sp, lens = s.block_table.cpu().to(torch.int64), s.seq_ptr.cpu().to(torch.int64), s.seq_lens.cpu()
    S = int(lens.numel())
    done, t, tokens = 0, 0.0, 0
    while done < min(max_seqs, S) and t < budget_s:
        pages = bt[sp[done]:sp[done + 1]]
        n = int(lens[done])
        kc = s.k_pool[pages.to(s.k_pool.device)].cpu()
        vc = s.v_pool[pages.to(s.v_pool.device)].cpu()
        local = torch.arange(pages.numel(), dtype=torch.int32)
        seq_ptr = torch.tensor([0, pages.numel()], dtype=torch.int32)
        token_ptr = torch.tensor([0, n], dtype=torch.int64)
        q = s.q[done:done + 1].cpu()
        t0 = time.perf_counter()
        for pool in (kc, vc):
            orc.unpack_block_paged(pool, local, seq_ptr, token_ptr, index_dtype=torch.int32)
        orc.paged_attention_decode(q, kc, vc, local[None, :], torch.tensor([n], dtype=torch.int32), s.scale)
        t += time.perf_counter() - t0
        tokens += n
        done += 1
    nbytes = step_bytes_total * tokens / s.total_tokens
    return nbytes / t / 1e9, t, done, nbytes


def run_csr(args, world, rank, local):
    """Bench line of the prefix-shared CSR workload: unpack K and V plus decode
    attention over the snapshot's pages, per step."""
    import pagedattention_decode_pkv_gb300 as pkv

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    cfg = wl.CONFIGS[args.config]
    step = CsrStep(pkv, cfg, seed=args.seed + rank, device=device)
    stream = torch.cuda.Stream(device)
    ptr = ctypes.c_void_p(stream.cuda_stream)
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step.run(ptr)
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    total_ms, (tw0, tw1) = time_graphs(step, args.steps, world)
    clocks = sampler.summary(tw0, tw1)
    sampler.stop()
    torch.cuda.synchronize()
    err = int(step.err.item())
    if err:
        raise RuntimeError(f"device error bits {err:#x} during the benchmark")
    per = time_csr_kernels(step, args.steps, world, stream)
    io, h2d, d2h = e2e_io(step)
    e2e_ms, _ = time_graphs(step, args.steps, world, io)

    total_ms_max = reduce_max(total_ms, world, device)
    e2e_ms_max = reduce_max(e2e_ms, world, device)
    all_bytes = reduce_sum(sum(step.bytes.values()) * args.steps, world, device)
    all_logical = reduce_sum(sum(step.logical.values()) * args.steps, world, device)
    value = all_bytes / (total_ms_max * 1e-3) / 1e9
    peak, peak_kind = measured_hbm_peak()
    unpack_ms = reduce_max((per["unpack_k"] + per["unpack_v"]) / 2, world, device)
    unpack_gbs = step.bytes["unpack_k"] / (unpack_ms * 1e-3) / 1e9
    attn_ms = reduce_max(per["paged_attention_decode"], world, device)

    cpu_baseline = None
    if world == 1 and not args.skip_cpu_baseline:
        gbs, secs, nseq, nbytes = csr_oracle_run(step.snap, sum(step.bytes.values()), step.S, args.cpu_budget_s)
        cpu_baseline = {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                        "sample": f"first {nseq} of {step.S} sequences, each unpacked (K and V) and attended alone "
                                  f"in {secs:.1f} s, single-threaded C oracle in binary64; bytes are those "
                                  f"sequences' token share of the pass's unique bytes ({nbytes / 1e9:.3f} GB)"}

    if rank != 0:
        return 0
    per_us = {k: round(v * 1e3, 2) for k, v in per.items()}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": round(total_ms_max / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_NAME[cfg.dtype],
        "data": "synthetic (seeded N(0,1) pools and q, randomly permuted pages, half the sequences aliasing one "
                "1024-token prefix)",
        "config": {
            "workload": cfg.name, "description": cfg.description, "num_seqs": step.S,
            "num_heads": cfg.num_heads, "head_dim": cfg.head_dim, "page_size": cfg.page_size,
            "total_tokens": step.T, "unique_tokens": step.unique_tokens, "nnz": step.nnz,
            "pages": step.num_pages,
            "step": "unpack K + unpack V (u32 CSR index buffers) + paged_attention_decode (+combine) over the "
                    "padded table",
            "step_bytes": sum(step.bytes.values()), "step_bytes_logical": sum(step.logical.values()),
            "l2": f"outputs of {2 * step.out_k.numel() * step.out_k.element_size() / 1e9:.2f} GB per step vs "
                  "129 MB L2; no flush",
            "parallelism": f"replicas x{world} (independent snapshots per rank, no data-path collective)",
        },
        "value_logical": round(all_logical / (total_ms_max * 1e-3) / 1e9, 2),
        "kernel_us": per_us,
        "kernel_gbs": {k: round(step.bytes[k] / (per[k] * 1e-3) / 1e9, 1) for k in per},
        "kernel_gbs_logical": {k: round(step.logical[k] / (per[k] * 1e-3) / 1e9, 1) for k in per},
        "roofline": {"kernel": "pkv_unpack_block_paged (per role)", "bound": "hbm",
                     "achieved": round(unpack_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(unpack_gbs / peak, 4), "peak_kind": peak_kind, "traffic": None,
                     "us_per_call": round(unpack_ms * 1e3, 2)},
        "attention": {"us_per_call": round(attn_ms * 1e3, 2),
                      "gbs_unique": round(step.bytes["paged_attention_decode"] / (attn_ms * 1e-3) / 1e9, 1),
                      "gbs_logical": round(step.logical["paged_attention_decode"] / (attn_ms * 1e-3) / 1e9, 1),
                      "decode_tokens_per_s": round(step.S / (attn_ms * 1e-3), 1)},
        "cpu_baseline": cpu_baseline,
        "e2e": {"value": round(all_bytes / (e2e_ms_max * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms_max / args.steps, 4)},
        "gpu_launches": 4 * args.steps,
        "timing": {"value": f"CUDA graphs of {STEPS_PER_GRAPH} passes replayed until `steps` passes ran between "
                            "two CUDA events; value counts unique bytes (each page row read once, every output "
                            "row written), value_logical every row a sequence names",
                   "kernel_us": "second pass: eager passes with CUDA events between the kernels, a 512 MB read "
                                "before each pass (outside the events) evicts L2",
                   "e2e": "graphs of the same passes as a pipelined loop runs them: q and the index buffers copied "
                          "from pinned host memory each pass as one packed buffer (two device input sets, copies on "
                          "a second stream), the attention output and error flag read back"},
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0



def run_reference_csr(args, world, rank):
    """The oracle as it stands on the CSR workload: two sequences per step,
    each unpacked (K and V) and attended alone; no library call."""
    if rank != 0:
        return 0
    cfg = wl.CONFIGS[args.config]
    device = "cuda" if torch.cuda.is_available() else "cpu"
    snap = wl.csr_snapshot(cfg, seed=args.seed, device=device)
    unique, _, _ = csr_step_bytes(cfg, snap)
    total = sum(unique.values())
    per_step = 2
    t, nbytes = 0.0, 0.0
    for i in range(args.warmup + args.steps):
        sub = csr_sub_snapshot(snap, i * per_step % cfg.num_seqs, per_step)
        _, dt, _, nb = csr_oracle_run(sub, total * sub.total_tokens / snap.total_tokens, per_step, 1e9)
        if i >= args.warmup:
            t += dt
            nbytes += nb
    value = nbytes / t / 1e9
    sample = (f"{per_step} sequences of the {cfg.name} snapshot per step, each unpacked (K and V) and attended "
              "alone; single-threaded C oracle in binary64; bytes are their token share of the pass's unique bytes")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_NAME[cfg.dtype],
        "data": "synthetic (seeded N(0,1), randomly permuted pages, aliased prefix)",
        "config": {"workload": cfg.name, "description": cfg.description, "num_seqs": cfg.num_seqs,
                   "l2": "bounded CPU sample; no GPU work"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def csr_sub_snapshot(snap, first: int, count: int):
    """Sequences [first, first + count) of a CSR snapshot as a snapshot of
    their own (same pools; index buffers rebased)."""
    from dataclasses import replace

    sp = snap.seq_ptr.cpu().to(torch.int64)
    lens = snap.seq_lens.cpu()[first:first + count]
    bt = snap.block_table.cpu()[sp[first]:sp[first + count]]
    new_sp = (sp[first:first + count + 1] - sp[first]).to(snap.seq_ptr.dtype)
    tp = torch.zeros(count + 1, dtype=torch.int64)
    tp[1:] = torch.cumsum(lens.to(torch.int64), 0)
    return replace(snap, block_table=bt, seq_ptr=new_sp, token_ptr=tp, seq_lens=lens,
                   block_tables_2d=snap.block_tables_2d.cpu()[first:first + count],
                   q=snap.q[first:first + count])

def run_profile_calls(args, local):
    """One kernel's calls on the workload (--profile-calls), for an ncu capture of a few launches."""
    import pagedattention_decode_pkv_gb300 as pkv

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    step = DecodeStep(pkv, wl.CONFIGS[args.config], seed=args.seed, device=device)
    call = step.attention
    if args.profile_calls in ("fp8", "int8"):
        step.make_codes(args.profile_calls)
        call = step.code8_attention
    elif args.profile_calls == "prefill":
        call = prefill_call(step)[0]
    elif args.profile_calls == "unpack":
        step._unpack_buffers()
        L, s, c, p = pkv._lib, step.snap, step.cfg, (lambda t: t.data_ptr())

        def call(ptr):
            return L.pkv_unpack_block_paged(p(step.unpacked_k), p(step.batch.k_cache), p(s.block_table),
                                            p(s.seq_ptr), pkv.PKV_U32, p(s.token_ptr), step.B, s.nnz, c.block_size,
                                            step.nb, c.num_kv_heads, c.head_dim, s.total_tokens, step.dt,
                                            p(step.err), ptr)
    elif args.profile_calls == "store":
        # every context token's row, scattered to its own slot (a prefill's store)
        L, b, c, p = pkv._lib, step.batch, step.cfg, (lambda t: t.data_ptr())
        bt, ctx, bs = b.block_tables.cpu(), step.ctx_cpu, c.block_size
        slots = torch.cat([bt[i, torch.arange(int(n)) // bs].to(torch.int64) * bs + torch.arange(int(n)) % bs
                           for i, n in enumerate(ctx)]).to(torch.int32).to(device)
        T = slots.numel()
        key = torch.randn(T, c.num_kv_heads, c.head_dim, device=device).to(c.dtype)
        value = torch.randn_like(key)
        step.profile_buffers = (slots, key, value)

        def call(ptr):
            return L.pkv_store_kvcache(p(key), p(value), p(b.k_cache), p(b.v_cache), p(slots), T, c.num_kv_heads,
                                       c.head_dim, step.nb * bs, step.dt, p(step.err), ptr)
    ptr = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(args.steps):
        if call(ptr) != 0:
            raise RuntimeError("pkv call failed: " + pkv._lib.pkv_last_error_string().decode())
    torch.cuda.synchronize()
    if int(step.err.item()):
        raise RuntimeError(f"device error bits {int(step.err.item()):#x}")
    print(f"{args.steps} {args.profile_calls} calls on {args.config}", flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_init(args)
    try:
        if args.config in CSR_CONFIGS:
            if args.impl == "reference":
                return run_reference_csr(args, world, rank)
            if args.profile_calls:
                raise SystemExit("--profile-calls takes a decode workload")
            return run_csr(args, world, rank, local)
        if args.impl == "reference":
            return run_reference(args, world, rank)
        if args.profile_calls:
            return run_profile_calls(args, local)
        return run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
