#!/usr/bin/env python
"""Benchmark of the MSA forward pass (libmsa) on GB300.

One step = the whole hot path (index scoring, block max-pooling, top-16 with
the local block forced, sparse softmax attention) over one batch of seeded
synthetic inputs already resident in HBM.  The default line is the 1M-token
chunked prefill, with the 128K single-call prefill and the 64 x 256K decode
batch measured in the same run and nested under "prefill_128k" and "decode":

  decode_256k   64 sequences x 262144-token block-major caches, 1 new query
                each (48 query / 8 KV heads, D 128, Di 64)
  prefill_128k  one 131072-token sequence, one call
  prefill_1m    one 1,048,576-token sequence, 128 chunked calls of 8192 queries
  prefill_32k   one 32768-token sequence
  decode_small  8 x 131072 decode (a small case for profiler captures)
  prefill_1m_last_chunk  the last 8192-query chunk of prefill_1m alone (profiling)
  dense_32k     dense causal attention over a 32768-token prefill (msa_dense_attn)
  decode_256k_paged  the decode batch from paged pools: the newest token of
                each sequence appended through a shuffled block table
                (msa_cache_append), then msa_forward_paged

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle (the
reference arm) on a bounded sample of the same workload instead.
"""
import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MSA prefill & decode tokens/s at 128K–1M ctx; % of TC/HBM roofline"
H, G, D, DI, BLK = 48, 8, 128, 64, 128
WORKLOADS = {
    "prefill_32k": dict(cfg=1, kind="prefill", B=1, L=32768, chunk=32768),
    "prefill_128k": dict(cfg=2, kind="prefill", B=1, L=131072, chunk=131072),
    "decode_256k": dict(cfg=3, kind="decode", B=64, L=262144),
    "prefill_1m": dict(cfg=4, kind="prefill", B=1, L=1048576, chunk=8192),
    # profiling cases (small enough for full profiler captures):
    # decode shapes at 8 x 131072 (K_idx 134 MB > L2, ~4 GB on device), and the
    # last 8192-query chunk of the 1M prefill alone (~4.5 GB on device)
    "decode_small": dict(cfg=3, kind="decode", B=8, L=131072),
    "prefill_1m_last_chunk": dict(cfg=4, kind="prefill", B=1, L=1048576, chunk=8192,
                                  only_last=True),
    # the rows built next to the path, measured on the same shapes:
    # dense causal attention over a 32K prefill (msa_dense_attn), and the
    # decode batch served from paged pools (msa_cache_append of the new token,
    # then msa_forward_paged through a shuffled block table)
    "dense_32k": dict(cfg=1, kind="prefill", B=1, L=32768, chunk=32768, mode="dense"),
    "decode_256k_paged": dict(cfg=3, kind="decode", B=64, L=262144, mode="paged"),
}
DEFAULT_WORKLOAD = "prefill_1m"
# queries per attention call when the e2e leg splits a single long prefill
E2E_SLICE = 8192
# most untimed e2e warm-up steps (they stop once two consecutive ones agree)
E2E_SETTLE_STEPS = 8
# oracle time the cpu_baseline figure accumulates (its sample is repeated)
CPU_BASELINE_SECONDS = 10.0
# measured in the same run and nested in the default line, under these keys
DEFAULT_SECONDARY = ("prefill_128k", "decode_256k")
NESTED_KEY = {"prefill_128k": "prefill_128k", "decode_256k": "decode"}


# ------------------------------------------------------------ algorithmic work --
def lb_of(t):
    return t // BLK


def attended_tokens(t):
    """Tokens the main branch attends for query position(s) t."""
    t = np.asarray(t, np.int64)
    return np.where(t < 16 * BLK, t + 1, 15 * BLK + t % BLK + 1)


def index_flops(t):
    """2*Di*G per scored (query, group, key); keys = the lb*128 candidate tokens."""
    t = np.asarray(t, np.int64)
    return float(np.sum(2.0 * DI * G * BLK * (t // BLK)))


def attn_flops(t):
    return float(np.sum(4.0 * D * H * attended_tokens(t)))


def dense_flops(t):
    """Dense causal attention: 4*D*H per (query, token <= t)."""
    return float(np.sum(4.0 * D * H * (np.asarray(t, np.int64) + 1)))


def decode_bytes(B, L):
    t = L - 1
    kidx = B * lb_of(t) * BLK * DI * 2                     # candidate blocks' K_idx
    kv = B * G * int(attended_tokens(t)) * D * 2 * 2       # gathered K and V
    small = B * (H * D * 2 * 2 + G * DI * 2 + G * 16 * 4)  # q, out, q_idx, sel
    return kidx, kv + small


# --------------------------------------------------------------------- clocks --
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu):
        self.rows, self.proc = [], None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if not self.rows:
            return None
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in self.rows for k in range(4)
                          if r[5 + k].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "fallback"


# ------------------------------------------------------------- distributed --
def dist_setup(gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    # NCCL reduces device tensors; gloo (the CPU test of this path) host ones
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ GPU arm --
class Job:
    """Device inputs and the sequence of C-ABI calls that make one step."""

    def __init__(self, name, rank):
        import torch
        import block_sparse_attention_04_gb300 as msa
        import msa_synth.device as sd
        self.msa = msa
        self.name, self.w = name, WORKLOADS[name]
        w = self.w
        self.B, self.L = w["B"], w["L"]
        self.nb = self.L // BLK
        self.seed = 20261202 + w["cfg"]
        b0 = rank * self.B
        if w["kind"] == "decode":
            self.calls = [dict(T=1, q_start=[self.L - 1] * self.B, kv_len=[self.L] * self.B,
                               qoff=0)]
            qrows = (self.L - 1, self.L)
        else:
            c = w["chunk"]
            starts = [self.L - c] if w.get("only_last") else list(range(0, self.L, c))
            self.calls = [dict(T=c, q_start=[s], kv_len=[s + c], qoff=s - starts[0])
                          for s in starts]
            qrows = (starts[0], self.L)
        self.dev = sd.make_inputs(self.B, H, G, D, DI, self.nb, self.L, self.seed, q_rows=qrows,
                                  b0=b0)
        T = self.calls[0]["T"]
        self.mode = w.get("mode", "sparse")
        self.params = msa.params(self.B, T, H, G, D, DI, self.nb)
        self.ws = msa.dense_workspace(self.params) if self.mode == "dense" else \
            msa.workspace(self.params)
        if self.mode == "paged":
            # the caches become one pool of B * nb blocks behind a shuffled
            # table; the newest token of each sequence is appended every step
            g = torch.Generator().manual_seed(self.seed)
            self.npool = self.B * self.nb
            self.table = torch.randperm(self.npool, generator=g).to(torch.int32).reshape(
                self.B, self.nb).cuda()
            pos = self.L - 1
            rows = self.table[:, pos // BLK].long() * BLK + pos % BLK
            self.k_new = self.dev["k"].reshape(-1, G, D)[rows].reshape(self.B, 1, G, D).clone()
            self.v_new = self.dev["v"].reshape(-1, G, D)[rows].reshape(self.B, 1, G, D).clone()
            self.kidx_new = self.dev["k_idx"].reshape(-1, DI)[rows].reshape(self.B, 1, DI).clone()
        self.sel = torch.empty((self.B, qrows[1] - qrows[0], G, 16), dtype=torch.int32,
                               device="cuda")
        self.out = torch.empty((self.B, qrows[1] - qrows[0], H, D), dtype=torch.int16,
                               device="cuda")
        torch.cuda.synchronize()

    def views(self, c, dev=None, sel=None, out=None):
        dev = dev or self.dev
        sel = self.sel if sel is None else sel
        out = self.out if out is None else out
        a, T = c["qoff"], c["T"]
        return (dev["q_idx"][:, a:a + T], dev["k_idx"], dev["q"][:, a:a + T], dev["k"], dev["v"],
                sel[:, a:a + T], out[:, a:a + T])

    def call(self, c):
        """Enqueue one call of the step (both entry points) on the current stream."""
        q_idx, k_idx, q, k, v, sel, out = self.views(c)
        self.msa.msa_index_topk(self.params, q_idx, k_idx, c["q_start"], c["kv_len"], sel, self.ws)
        self.msa.msa_sparse_attn(self.params, q, k, v, sel, c["q_start"], c["kv_len"], out, self.ws)

    def step(self, ev=None):
        """Enqueue one step; ev: list to which (start, mid, end) events are appended."""
        import torch
        msa = self.msa
        if self.mode != "sparse":
            return self.step_other(ev)
        for c in self.calls:
            q_idx, k_idx, q, k, v, sel, out = self.views(c)
            if ev is not None:
                e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                e[0].record()
            msa.msa_index_topk(self.params, q_idx, k_idx, c["q_start"], c["kv_len"], sel, self.ws)
            if ev is not None:
                e[1].record()
            msa.msa_sparse_attn(self.params, q, k, v, sel, c["q_start"], c["kv_len"], out,
                                self.ws)
            if ev is not None:
                e[2].record()
                ev.append(e)

    def step_other(self, ev):
        """Dense attention, or the paged decode step (append, then forward)."""
        import torch
        msa = self.msa
        for c in self.calls:
            q_idx, k_idx, q, k, v, sel, out = self.views(c)
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)] if ev is not None else None
            if e:
                e[0].record()
            if self.mode == "paged":
                msa.msa_cache_append(self.params, self.k_new, self.v_new, self.kidx_new,
                                     c["q_start"], k, v, k_idx, self.ws, block_table=self.table,
                                     num_pool_blocks=self.npool)
            if e:
                e[1].record()
            if self.mode == "dense":
                msa.msa_dense_attn(self.params, q, k, v, c["q_start"], c["kv_len"], out, self.ws)
            else:
                msa.msa_forward_paged(self.params, self.table, self.npool, q_idx, k_idx, q, k, v,
                                      c["q_start"], c["kv_len"], out, self.ws, sel_out=sel)
            if e:
                e[2].record()
                ev.append(e)

    def tokens(self):
        return self.B * sum(c["T"] for c in self.calls)

    def positions(self):
        if self.w["kind"] == "decode":
            return np.full(self.B, self.L - 1, np.int64)
        return np.concatenate([np.arange(c["q_start"][0], c["q_start"][0] + c["T"], dtype=np.int64)
                               for c in self.calls])


def selection_quality(job, nrows, seed=7):
    """Attention-mass coverage and selection recall of the step's selections
    (msa_selection_quality) on nrows seeded query positions; not timed."""
    import torch
    msa = job.msa
    rng = np.random.default_rng(seed)
    if job.w["kind"] == "decode":
        calls = [(job.B, 0, [job.L - 1] * job.B)]
    else:
        pos = job.positions()
        pick = np.sort(rng.choice(len(pos), size=min(nrows, len(pos)), replace=False))
        calls = [(1, int(a), [int(pos[a])]) for a in pick]
    cov, best, rec = [], [], []
    for B, a, qs in calls:
        p = msa.params(B, 1, H, G, D, DI, job.nb)
        ws = msa.quality_workspace(p)
        c = torch.empty((B, 1, H), dtype=torch.float32, device="cuda")
        bc = torch.empty_like(c)
        ds = torch.empty((B, 1, G, 16), dtype=torch.int32, device="cuda")
        hits = torch.empty((B, 1, G), dtype=torch.int32, device="cuda")
        msa.msa_selection_quality(p, job.dev["q"][:, a:a + 1], job.dev["k"], job.sel[:, a:a + 1],
                                  qs, [t + 1 for t in qs], c, bc, ds, hits, ws)
        nsel = np.minimum(16, np.asarray(qs) // BLK + 1)[:, None, None]
        cov.append(c.cpu().numpy().reshape(-1))
        best.append(bc.cpu().numpy().reshape(-1))
        rec.append((hits.cpu().numpy() / nsel).reshape(-1))
    cov, best, rec = np.concatenate(cov), np.concatenate(best), np.concatenate(rec)
    return {"rows": len(calls) if job.w["kind"] != "decode" else job.B,
            "coverage_mean": float(cov.mean()), "coverage_min": float(cov.min()),
            "best_coverage_mean": float(best.mean()), "recall_mean": float(rec.mean()),
            "recall_min": float(rec.min()),
            "definition": "coverage: full causal softmax mass inside the 16 selected blocks, "
                          "per (query, head); best: the same for the ideal selection (local "
                          "block + top-15 by group-averaged mass); recall: |selected and "
                          "ideal| / |ideal| per (query, group)"}


def capture_step(job):
    """One step of `job` captured into a CUDA graph (the C-ABI calls enqueue
    kernels and memsets only, so they capture as they are), or None if the
    capture fails."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    try:
        with torch.cuda.stream(side):
            job.step()                      # settles lazy per-function attributes
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            job.step()
        torch.cuda.synchronize()
        return g
    except RuntimeError:
        torch.cuda.synchronize()
        return None


def time_job(job, steps, warmup, world, graph=True):
    """Warm-up, then two timed passes of `steps` steps each.  The eager pass
    enqueues every call from Python with events around the index and attention
    calls (their split, and the kernel count).  The headline pass replays the
    same step captured into a CUDA graph, as a serving loop would, so that the
    step is timed without per-call launch gaps; with graph=False (or if the
    capture fails) the eager pass is the headline."""
    import torch
    for _ in range(warmup):
        job.step()
    job.msa.msa_workspace_status(job.ws)
    torch.cuda.synchronize()
    n0 = job.msa.msa_kernel_launch_count()
    barrier(world)
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    time.sleep(0.3)
    ev = []
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        job.step(ev)
    t1.record()
    torch.cuda.synchronize()
    barrier(world)
    launches = job.msa.msa_kernel_launch_count() - n0
    job.msa.msa_workspace_status(job.ws)
    eager_ms = max_over_ranks(t0.elapsed_time(t1), world)
    idx_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / steps
    att_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / steps
    g = capture_step(job) if graph else None
    total_ms, mode = eager_ms, "eager"
    if g is not None:
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        job.msa.msa_workspace_status(job.ws)
        barrier(world)
        torch.cuda.synchronize()
        t0.record()
        for _ in range(steps):
            g.replay()
        t1.record()
        torch.cuda.synchronize()
        barrier(world)
        job.msa.msa_workspace_status(job.ws)
        total_ms, mode = max_over_ranks(t0.elapsed_time(t1), world), "cuda graph"
        del g
    ck = clocks.stop()
    return {"total_ms": total_ms, "eager_ms": eager_ms, "idx_ms": idx_ms, "att_ms": att_ms,
            "launches": launches, "clocks": ck, "mode": mode}


class HostBuffers:
    """Page-locked host tensors for the e2e leg.

    kind "thp": anonymous memory advised onto transparent huge pages (the
    host's PMD size), aligned to that size, then page-locked with
    cudaHostRegister, so that a copy walks few, large physical runs; kind
    "torch": torch's pinned allocator (cudaHostAlloc); kind "auto": a "thp"
    buffer, kept if a copy of all of it runs at AUTO_MIN_GBS or more (or it
    is small), else the faster of it and a "torch" buffer (after a long run
    of other work the host's free memory can be so scattered that either
    kind copies slowly)."""

    AUTO_MIN_GBS = 150.0
    AUTO_MIN_BYTES = 256 << 20          # smaller copies are latency-bound: not probed

    def __init__(self, kind):
        self.kind, self.maps, self.regs = kind, [], []
        self.used = []                  # the kind each buffer ended up with
        self.probed = {"h2d": [], "d2h": []}  # GB/s of the buffers kept
        self.huge = 2 << 20
        try:
            with open("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size") as f:
                self.huge = int(f.read())
        except (OSError, ValueError):
            pass

    def empty(self, shape, dtype, to_device=True):
        """to_device: the buffer is a copy source (H2D) rather than a target."""
        import torch
        if self.kind == "torch":
            self.used.append("torch")
            return torch.empty(shape, dtype=dtype, pin_memory=True)
        t = self._thp(shape, dtype)
        kind = "thp"
        if self.kind == "auto" and t.numel() * t.element_size() >= self.AUTO_MIN_BYTES:
            bw = self._probe(t, to_device)
            if bw < self.AUTO_MIN_GBS:
                t2 = torch.empty(shape, dtype=dtype, pin_memory=True)
                bw2 = self._probe(t2, to_device)
                if bw2 > bw:
                    self._unregister(t.data_ptr())
                    del t
                    self.maps.pop()         # the mapping goes once nothing views it
                    t, kind, bw = t2, "torch", bw2
            self.probed["h2d" if to_device else "d2h"].append(bw)
        self.used.append(kind)
        return t

    def _thp(self, shape, dtype):
        import mmap
        import torch
        item = torch.empty((), dtype=dtype).element_size()
        n = int(np.prod(shape)) * item
        span = (n + 2 * self.huge - 1) // self.huge * self.huge
        m = mmap.mmap(-1, span, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
        base = np.frombuffer(m, dtype=np.uint8)
        off = (-base.ctypes.data) % self.huge
        try:
            m.madvise(mmap.MADV_HUGEPAGE, off, span - off)
        except (AttributeError, OSError, ValueError):
            pass
        t = torch.frombuffer(m, dtype=dtype, count=n // item, offset=off).view(shape)
        rc = torch.cuda.cudart().cudaHostRegister(t.data_ptr(), n, 0)
        if int(rc) != 0:
            raise RuntimeError("cudaHostRegister failed (%s)" % rc)
        self.maps.append((m, base))
        self.regs.append(t.data_ptr())
        return t

    @staticmethod
    def _probe(t, to_device, chunk=1 << 30):
        """Copy bandwidth (GB/s) of the whole of t (page placement differs
        along a buffer), in copies of up to `chunk` bytes."""
        import torch
        flat = t.view(-1).view(torch.uint8)
        n = min(flat.numel(), chunk)
        d = torch.empty(n, dtype=torch.uint8, device="cuda")
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for a in range(0, flat.numel(), chunk):
            h = flat[a:a + chunk]
            if to_device:
                d[:h.numel()].copy_(h, non_blocking=True)
            else:
                h.copy_(d[:h.numel()], non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        del d
        return flat.numel() / (e0.elapsed_time(e1) / 1e3) / 1e9

    def _unregister(self, ptr):
        import torch
        torch.cuda.cudart().cudaHostUnregister(ptr)
        self.regs.remove(ptr)

    def describe(self):
        kinds = {"thp": "page-locked transparent huge pages", "torch": "torch pinned allocator"}
        used = sorted(set(self.used))
        return " + ".join(kinds[k] for k in used) if used else kinds.get(self.kind, self.kind)

    def release(self):
        import torch
        for ptr in self.regs:
            torch.cuda.cudart().cudaHostUnregister(ptr)
        self.regs = []


def time_e2e(job, steps, world, host_alloc="auto", graph=True):
    """Same step through the C ABI with host buffers: pinned H2D of the step's
    inputs and D2H of its outputs inside the timed region."""
    import torch
    if job.w["kind"] == "decode":
        names = ["q_idx", "q"]      # the caches stay resident between decode steps
    else:
        names = ["q_idx", "k_idx", "q", "k", "v"]
    bufs = HostBuffers(host_alloc)
    host = {n: bufs.empty(job.dev[n].shape, torch.int16) for n in names}
    for n in names:
        host[n].copy_(job.dev[n])
    sel_h = bufs.empty(job.sel.shape, torch.int32, to_device=False)
    out_h = bufs.empty(job.out.shape, torch.int16, to_device=False)
    h2d = sum(host[n].numel() * 2 for n in names)
    d2h = sel_h.numel() * 4 + out_h.numel() * 2
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    prefill = job.w["kind"] != "decode" and job.B == 1 and job.mode == "sparse"
    pipelined = prefill and len(job.calls) > 1
    # A single long prefill call: one index call over all its queries, then
    # the attention as consecutive calls of E2E_SLICE queries each (the same
    # kernels and results as one call, which runs in passes of that length),
    # so that the query rows go up and the outputs come back while other
    # slices compute.
    sliced = prefill and len(job.calls) == 1 and job.calls[0]["T"] > E2E_SLICE
    if pipelined or sliced:
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    else:
        side_in, side_out = torch.cuda.Stream(), torch.cuda.Stream()
    if sliced:
        c0 = job.calls[0]
        slice_params = job.msa.params(1, E2E_SLICE, H, G, D, DI, job.nb)
        tail = c0["T"] % E2E_SLICE
        tail_params = job.msa.params(1, tail, H, G, D, DI, job.nb) if tail else None

    def record(stream):
        e = torch.cuda.Event()
        e.record(stream)
        return e

    def run_sliced(n):
        c = c0
        st, T = c["q_start"][0], c["T"]
        msa = job.msa
        comp = torch.cuda.current_stream()
        for _ in range(n):
            s_in.wait_stream(comp)      # steps do not overlap
            with torch.cuda.stream(s_in):
                job.dev["q_idx"].copy_(host["q_idx"], non_blocking=True)
                job.dev["k_idx"].copy_(host["k_idx"], non_blocking=True)
                ev_idx = record(s_in)
                job.dev["k"].copy_(host["k"], non_blocking=True)
                job.dev["v"].copy_(host["v"], non_blocking=True)
                ev_q = []
                for a in range(0, T, E2E_SLICE):
                    job.dev["q"][:, a:a + E2E_SLICE].copy_(host["q"][:, a:a + E2E_SLICE],
                                                           non_blocking=True)
                    ev_q.append(record(s_in))
            comp.wait_event(ev_idx)
            msa.msa_index_topk(job.params, job.dev["q_idx"], job.dev["k_idx"], c["q_start"],
                               c["kv_len"], job.sel, job.ws)
            ev_sel = record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_sel)
                sel_h.copy_(job.sel, non_blocking=True)
            for j, a in enumerate(range(0, T, E2E_SLICE)):
                n_j = min(E2E_SLICE, T - a)
                comp.wait_event(ev_q[j])    # after K/V, on the same stream
                msa.msa_sparse_attn(slice_params if n_j == E2E_SLICE else tail_params,
                                    job.dev["q"][:, a:a + n_j], job.dev["k"], job.dev["v"],
                                    job.sel[:, a:a + n_j], [st + a], c["kv_len"],
                                    job.out[:, a:a + n_j], job.ws)
                ev_o = record(comp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_o)
                    out_h[:, a:a + n_j].copy_(job.out[:, a:a + n_j], non_blocking=True)
            comp.wait_stream(s_out)

    def run(n):
        if sliced:
            run_sliced(n)
            return
        if not pipelined:
            # one call: the index inputs go up first; the attention's inputs
            # follow on a side stream while the index call runs, and sel comes
            # back on another while the attention runs
            cur = torch.cuda.current_stream()
            first = [nm for nm in ("q_idx", "k_idx") if nm in names]
            rest = [nm for nm in names if nm not in first]
            (c,) = job.calls
            q_idx, k_idx, q, k, v, sel, out = job.views(c)
            for _ in range(n):
                for nm in first:
                    job.dev[nm].copy_(host[nm], non_blocking=True)
                side_in.wait_stream(cur)
                with torch.cuda.stream(side_in):
                    for nm in rest:
                        job.dev[nm].copy_(host[nm], non_blocking=True)
                job.msa.msa_index_topk(job.params, q_idx, k_idx, c["q_start"], c["kv_len"], sel,
                                       job.ws)
                side_out.wait_stream(cur)
                with torch.cuda.stream(side_out):
                    sel_h.copy_(job.sel, non_blocking=True)
                cur.wait_stream(side_in)
                job.msa.msa_sparse_attn(job.params, q, k, v, sel, c["q_start"], c["kv_len"], out,
                                        job.ws)
                out_h.copy_(job.out, non_blocking=True)
                cur.wait_stream(side_out)
            return
        # chunked prefill, pipelined as a caller of the C ABI would run it:
        # chunk c's inputs (its q_idx and q rows, the k_idx rows and K/V blocks
        # of its own 8192 tokens) go up on one stream, its call runs on the
        # compute stream once they have landed, and its out and sel rows come
        # back on a third stream while the next chunk computes.  The same
        # bytes move as in the serial form; only their overlap differs.
        comp = torch.cuda.current_stream()
        for _ in range(n):
            s_in.wait_stream(comp)      # steps do not overlap
            for c in job.calls:
                a, T, st = c["qoff"], c["T"], c["q_start"][0]
                kb0, kb1 = st // BLK, (st + T) // BLK
                with torch.cuda.stream(s_in):
                    job.dev["q_idx"][:, a:a + T].copy_(host["q_idx"][:, a:a + T], non_blocking=True)
                    job.dev["q"][:, a:a + T].copy_(host["q"][:, a:a + T], non_blocking=True)
                    job.dev["k_idx"][:, st:st + T].copy_(host["k_idx"][:, st:st + T],
                                                         non_blocking=True)
                    job.dev["k"][:, kb0:kb1].copy_(host["k"][:, kb0:kb1], non_blocking=True)
                    job.dev["v"][:, kb0:kb1].copy_(host["v"][:, kb0:kb1], non_blocking=True)
                    ev_in = torch.cuda.Event()
                    ev_in.record(s_in)
                comp.wait_event(ev_in)
                job.call(c)
                ev_done = torch.cuda.Event()
                ev_done.record(comp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_done)
                    sel_h[:, a:a + T].copy_(job.sel[:, a:a + T], non_blocking=True)
                    out_h[:, a:a + T].copy_(job.out[:, a:a + T], non_blocking=True)
            comp.wait_stream(s_out)

    # Untimed warm-up steps until two consecutive ones agree within 5 % (at
    # most E2E_SETTLE_STEPS): right after other heavy host-memory work (a
    # test suite) the host copies run slowly for some seconds.
    prev = None
    for _ in range(E2E_SETTLE_STEPS):
        w0 = torch.cuda.Event(enable_timing=True)
        w1 = torch.cuda.Event(enable_timing=True)
        w0.record()
        run(1)
        w1.record()
        torch.cuda.synchronize()
        cur = w0.elapsed_time(w1)
        if prev is not None and abs(cur - prev) <= 0.05 * cur:
            break
        prev = cur
    # A single call per step (decode, a prefill of one slice) is replayed as a
    # CUDA graph of its copies and calls, as a serving loop would run it; each
    # replay moves the same bytes.  The pipelined and sliced prefills stay
    # eager: replayed as graphs, their copies ran at a third of the speed of
    # the same eager copies in runs that followed the GPU test suite.
    g, mode = None, "eager"
    if graph and not pipelined and not sliced:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                run(1)
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            mode = "cuda graph"
        except RuntimeError:
            torch.cuda.synchronize()
            g = None
    barrier(world)
    t0.record()
    if g is not None:
        for _ in range(steps):
            g.replay()
    else:
        run(steps)
    t1.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1), world) / steps
    del g, host, sel_h, out_h
    described = bufs.describe()
    probed = {k: round(min(v), 1) for k, v in bufs.probed.items() if v}
    if probed:
        described += " (slowest buffer copied at %s GB/s)" % ", ".join(
            "%s %s" % (k, v) for k, v in sorted(probed.items()))
    bufs.release()
    if pipelined:
        mode += ", copies pipelined per chunk"
    elif sliced:
        mode += ", index call then attention in %d-query calls, copies pipelined" % E2E_SLICE
    else:
        mode += ", attention inputs up and sel down beside the calls"
    return ms, h2d, d2h, mode, described


# ---------------------------------------------------------------- CPU arm --
class OracleSample:
    """The CPU oracle on a bounded, seeded sample of workload `name`.

    Inputs are generated once (outside the timed region); run() times the
    oracle's selection and attention for the sampled query rows."""

    def __init__(self, name, rows=None, nthreads=None):
        import msa_synth as syn
        import oracle
        self.syn, self.oracle = syn, oracle
        w = WORKLOADS[name]
        self.seed = 20261202 + w["cfg"]
        self.nthreads = nthreads or (os.cpu_count() or 1)
        self.d = oracle.dims(H, G, D, DI)
        self.nb = w["L"] // BLK
        self.dense = w.get("mode") == "dense"
        rng = np.random.default_rng(self.seed)
        if w["kind"] == "decode":
            nseq = rows or 16
            t = w["L"] - 1
            self.rows = [(b, t) for b in range(nseq)]
            self.desc = ("%d of the 64 decode sequences (query at position %d), all groups "
                         "and heads" % (nseq, t))
        else:
            nrows = rows or 24
            ts = np.sort(rng.choice(w["L"], size=nrows, replace=False))
            self.rows = [(0, int(t)) for t in ts]
            self.desc = ("%d query positions drawn uniformly from the %d of the sequence, all "
                         "groups and heads" % (nrows, w["L"]))
        L = w["L"]
        self.kidx = {b: syn.kidx_seq(self.seed, b, L, DI) for b in sorted({b for b, _ in self.rows})}
        self.qidx = {r: syn.qidx_rows(self.seed, r[0], r[1], r[1] + 1, G, DI)[0] for r in self.rows}
        self.q = {r: syn.q_rows(self.seed, r[0], r[1], r[1] + 1, H, D)[0] for r in self.rows}
        self.kv = {}

    def _kv(self, row, sel):
        if row not in self.kv:
            syn = self.syn
            blocks = sorted({int(x) for x in sel.reshape(-1) if x >= 0})
            kc = np.zeros((self.nb, BLK, G, D), np.uint16)
            vc = np.zeros((self.nb, BLK, G, D), np.uint16)
            kc[blocks] = syn.kv_blocks(self.seed, syn.TID_K, row[0], blocks, G, D)
            vc[blocks] = syn.kv_blocks(self.seed, syn.TID_V, row[0], blocks, G, D)
            self.kv[row] = (kc, vc)
        return self.kv[row]

    def run(self):
        """Returns (tokens_per_s, timed seconds)."""
        from concurrent.futures import ThreadPoolExecutor
        o, d = self.oracle, self.d
        if self.dense:
            # dense attention over every token <= t (the caches, made once)
            if not self.kv:
                syn = self.syn
                self.kv[0] = (syn.kv_cache(self.seed, syn.TID_K, 0, self.nb, G, D),
                              syn.kv_cache(self.seed, syn.TID_V, 0, self.nb, G, D))
            kc, vc = self.kv[0]
            t0 = time.perf_counter()
            with ThreadPoolExecutor(self.nthreads) as ex:
                list(ex.map(lambda r: o.dense(d, r[1], self.q[r], kc, vc), self.rows))
            secs = time.perf_counter() - t0
            return len(self.rows) / secs, secs
        t0 = time.perf_counter()
        with ThreadPoolExecutor(self.nthreads) as ex:
            sels = list(ex.map(lambda r: o.select(d, r[1], self.qidx[r], self.kidx[r[0]]),
                               self.rows))
        secs = time.perf_counter() - t0
        kvs = [self._kv(r, s) for r, s in zip(self.rows, sels)]   # not timed
        t0 = time.perf_counter()
        with ThreadPoolExecutor(self.nthreads) as ex:
            list(ex.map(lambda a: o.attend(d, a[0][1], self.q[a[0]], a[1][0], a[1][1], a[2]),
                        zip(self.rows, kvs, sels)))
        secs += time.perf_counter() - t0
        return len(self.rows) / secs, secs


def reference_arm(args, world, rank):
    if rank != 0:
        return
    name = args.workload
    w = WORKLOADS[name]
    smp = OracleSample(name, rows=args.ref_rows)
    for _ in range(args.warmup):
        smp.run()
    vals, secs = [], 0.0
    for _ in range(args.steps):
        v, s = smp.run()
        vals.append(v)
        secs += s
    value = len(smp.rows) * args.steps / secs
    threads, desc = smp.nthreads, smp.desc
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * secs / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": name, "batch": w["B"], "ctx": w["L"], "heads": H,
                   "kv_heads": G, "head_dim": D, "index_dim": DI},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# DRAM traffic of the dominant kernel comes from a recorded ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum of one launch on a small case,
# scaled to this workload's launches by the algorithmic work), stored with a
# hash of the kernel sources it was taken on.  When those sources change, the
# figure no longer describes the kernel and `traffic` is reported as null.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")
KERNEL_SOURCES = {
    "index_tc": ["msa_index_tc.cu", "msa_device.cuh", "msa_internal.h"],
    "index_stream": ["msa_stream.cu", "msa_device.cuh", "msa_internal.h"],
}


def kernel_sources_sha(kernel):
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "block_sparse_attention_04_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, units_per_launch):
    """DRAM bytes per launch of `kernel` for a launch processing units_per_launch
    algorithmic units (flops or bytes), or None if no capture matches the
    current sources."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)[kernel]
    except (OSError, ValueError, KeyError):
        return None
    if rec.get("sources_sha") != kernel_sources_sha(kernel):
        return None
    return rec["dram_bytes"] * units_per_launch / rec["units"]


def measure(name, args, world, rank):
    """Time workload `name`; returns the fields of its JSON line."""
    import torch
    peaks, peak_kind = measured_peaks()
    job = Job(name, rank)
    tj = time_job(job, args.steps, args.warmup, world, graph=not args.no_graph)
    ms = tj["total_ms"] / args.steps
    idx_ms, att_ms, launches, clocks = tj["idx_ms"], tj["att_ms"], tj["launches"], tj["clocks"]
    tokens = job.tokens() * world
    w = job.w
    pos = job.positions()
    if job.mode == "dense":
        fa = dense_flops(pos) * job.B
        sustained = ms * args.steps > 1000
        peak_tf = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
        roof = {"bound": "tensor", "kernel": "dense attention (msa_dense_attn: dense_tc_kernel, "
                "query-outer with O in tensor memory)",
                "achieved": fa / (att_ms / 1000.0) / 1e12, "peak": peak_tf, "unit": "TFLOP/s",
                "traffic": None, "peak_kind": peak_kind + (" sustained" if sustained else " burst"),
                "flops_per_step": fa}
        roof["frac"] = roof["achieved"] / roof["peak"]
        whole = {"flops_per_step": fa, "achieved_tflops": fa / (ms / 1000.0) / 1e12}
    elif job.mode == "paged":
        kidx_b, rest_b = decode_bytes(job.B, job.L)
        app_b = job.B * 2 * (2 * G * D + DI) * 2     # read and write of the new rows
        step_b = kidx_b + rest_b + app_b
        roof = {"bound": "hbm", "kernel": "paged decode step (msa_cache_append + "
                "msa_forward_paged through the block table)",
                "achieved": step_b / (ms / 1000.0) / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "traffic": None, "peak_kind": peak_kind,
                "bytes_per_step": step_b}
        roof["frac"] = roof["achieved"] / roof["peak"]
        whole = {"bytes_per_step": step_b, "append_ms": idx_ms, "forward_ms": att_ms}
    elif w["kind"] == "decode":
        kidx_b, rest_b = decode_bytes(job.B, job.L)
        roof = {"bound": "hbm",
                "kernel": "index scan (msa_index_topk: index_stream + topk_merge)",
                "achieved": kidx_b / (idx_ms / 1000.0) / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "traffic": recorded_traffic("index_stream", kidx_b),
                "peak_kind": peak_kind,
                "bytes_per_launch": kidx_b}
        roof["frac"] = roof["achieved"] / roof["peak"]
        whole = {"bytes_per_step": kidx_b + rest_b,
                 "achieved_gbs": (kidx_b + rest_b) / (ms / 1000.0) / 1e9}
        whole["frac_of_hbm"] = whole["achieved_gbs"] / peaks["hbm_gbs"]
    else:
        fi = index_flops(pos) * job.B
        fa = attn_flops(pos) * job.B
        # a timed region of seconds runs under the power cap: sustained peak
        sustained = ms * args.steps > 1000
        peak_tf = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
        roof = {"bound": "tensor",
                "kernel": "index scan (msa_index_topk: index_tc + topk_merge)",
                "achieved": fi / (idx_ms / 1000.0) / 1e12, "peak": peak_tf, "unit": "TFLOP/s",
                "traffic": recorded_traffic("index_tc", fi / len(job.calls)),
                "peak_kind": peak_kind + (" sustained" if sustained else " burst"),
                "flops_per_step": fi, "launches_per_step": len(job.calls)}
        roof["frac"] = roof["achieved"] / roof["peak"]
        whole = {"flops_per_step": fi + fa, "index_flops": fi, "attn_flops": fa,
                 "achieved_tflops": (fi + fa) / (ms / 1000.0) / 1e12,
                 "attn_achieved_tflops": fa / (att_ms / 1000.0) / 1e12}
        whole["frac_of_bf16_peak"] = whole["achieved_tflops"] / peak_tf
    quality = selection_quality(job, args.quality_rows) \
        if args.quality_rows > 0 and job.mode == "sparse" else None
    if job.mode == "sparse":
        e2e_ms, h2d, d2h, e2e_mode, host_desc = time_e2e(job, max(1, min(args.steps, 3)), world,
                                                         args.host_alloc, graph=not args.no_graph)
    else:
        e2e_ms, h2d, d2h, e2e_mode, host_desc = None, 0, 0, None, None
    cfg = {"workload": name, "batch": job.B, "ctx": job.L, "calls_per_step": len(job.calls),
           "queries_per_call": job.calls[0]["T"], "heads": H, "kv_heads": G, "head_dim": D,
           "index_dim": DI, "block": BLK, "topk": 16, "l2": "inputs larger than L2 (no flush)",
           "launch": tj["mode"], "eager_ms_per_step": tj["eager_ms"] / args.steps}
    del job
    torch.cuda.empty_cache()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        # the sample is run again until about CPU_BASELINE_SECONDS of oracle
        # time have accumulated (bounded), so the figure is not one short burst
        smp = OracleSample(name)
        secs, passes = 0.0, 0
        while passes < 1 or (secs < CPU_BASELINE_SECONDS and passes < 200):
            secs += smp.run()[1]
            passes += 1
        cpu = {"value": len(smp.rows) * passes / secs, "unit": "tokens/s", "cores": smp.nthreads,
               "kind": "oracle", "sample": "%s; run %d times" % (smp.desc, passes),
               "seconds": secs}
    return {"value": tokens / (ms / 1000.0), "ms_per_step": ms, "config": cfg, "roofline": roof,
            "step": whole, "kernels_ms": {"index_topk": idx_ms, "sparse_attn": att_ms},
            "e2e": None if e2e_ms is None else {
                "value": tokens / (e2e_ms / 1000.0), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "host_buffers": host_desc,
                "launch": e2e_mode},
            "gpu_launches": int(launches), "clocks": clocks, "cpu_baseline": cpu,
            "selection_quality": quality}


def gpu_arm(args, world, rank):
    import block_sparse_attention_04_gb300 as msa
    msa.load()
    r = measure(args.workload, args, world, rank)
    line = {
        "metric": METRIC, "value": r["value"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded msa_synth generator: Irwin-Hall normals, 2^-3 index grid "
                "with needles)",
    }
    for k in ("config", "roofline", "step", "kernels_ms", "e2e", "gpu_launches", "clocks",
              "cpu_baseline", "selection_quality"):
        line[k] = r[k]
    for sec in args.secondary:
        if sec == args.workload:
            continue
        s = measure(sec, args, world, rank)
        line[NESTED_KEY.get(sec, sec)] = {
            "workload": sec, "value": s["value"], "unit": "tokens/s",
            "ms_per_step": s["ms_per_step"], "config": s["config"], "roofline": s["roofline"],
            "step": s["step"], "kernels_ms": s["kernels_ms"], "e2e": s["e2e"],
            "gpu_launches": s["gpu_launches"], "clocks": s["clocks"],
            "cpu_baseline": s["cpu_baseline"], "selection_quality": s["selection_quality"]}
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--ref-rows", type=int, default=None,
                    help="rows of the bounded oracle sample per reference step")
    ap.add_argument("--secondary", default=None,
                    help="comma-separated workloads reported in the same line (default: "
                         "prefill_128k,decode_256k when the workload is the default one; "
                         "'none' to skip)")
    ap.add_argument("--host-alloc", choices=["auto", "thp", "torch"], default="auto",
                    help="host buffers of the e2e leg: page-locked transparent huge pages, "
                         "torch's pinned allocator, or (default) huge pages unless a probe "
                         "copy shows the other kind faster")
    ap.add_argument("--quality-rows", type=int, default=64,
                    help="query positions sampled for the selection-quality figures (0: skip)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-graph", action="store_true",
                    help="time the eager step as the headline instead of its CUDA-graph replay")
    args = ap.parse_args()
    if args.secondary is None:
        args.secondary = ",".join(DEFAULT_SECONDARY) if args.workload == DEFAULT_WORKLOAD \
            else "none"
    args.secondary = [] if args.secondary == "none" else \
        [w for w in args.secondary.split(",") if w]
    for w in args.secondary:
        if w not in WORKLOADS:
            ap.error("unknown workload %r" % w)
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        import oracle
        oracle.build()
        reference_arm(args, world, rank)
        return
    from block_sparse_attention_04_gb300 import _build
    import msa_synth.device as sd
    _build.build()
    sd.build()
    world, rank, _ = dist_setup(args.gpus)
    gpu_arm(args, world, rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
