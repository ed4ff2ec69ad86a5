"""Benchmark of the paged FP8 KV decode hot path on GB300.

Headline step: 64 requests of 131,072 tokens each (64 query / 8 kv heads,
head dim 128, page size 16, FP8 e4m3 cache): every request appends its new
token's K/V (bf16 -> e4m3 with per-(page, kv-head) scales), the batched
page-tag check runs, then split-K decode attention and the combine.  `value`
is decode tokens/s with each step replayed as a CUDA graph; `roofline` is the
split phase against the measured HBM copy bandwidth (and split + combine with
Q and O counted, under `roofline.attn`).  The same line carries, under
`roofline.points`, the other configurations: the 1..32-request points and the
BF16 cache at 128k, the 32-request GQA batch (4k..32k), the skewed
256-request stress step, the 96 q / 8 kv group, the latent tensor-core
verify, the tag-check overhead (separate pass and fused), the bulk append and
the handoff from a BF16 pool; each step line gives the attention's GB/s from
CUDA events around an eager call and from its share of a CUDA-graph step
(`frac_graph`).  `cpu_baseline` is the
CPU oracle replaying sampled requests' first step, with the element-wise
comparison of the GPU's outputs for those requests (`parity`).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--detail FILE]

Prints one JSON line (rank 0); --detail also writes every measured line to a
file.  --impl reference times the CPU oracle, as it stands, on the headline
workload.  Multi-GPU runs are data-parallel replicas (one pool and one
request shard per rank, no collective on the data path); the step time is the
max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = ("decode attn tokens/s & achieved HBM GB/s vs ~8 TB/s, FP8 vs BF16 KV, 1×GB300")
NOMINAL_HBM_GBS = 8000.0

# DRAM bytes of gqa_split_kernel<e4m3> per launch from one ncu capture
# (dram__bytes_read.sum per algorithmic byte, dram__bytes_write.sum per
# (CTA, segment) piece), valid only while the kernel's sources hash to `sha`
# (sha256 of the listed files, first 16 hex digits); otherwise the line
# reports traffic null.
SPLIT_DRAM = {"sources": ["decode_gqa.cu", "decode_plan.cuh", "common.cuh"],
              "sha": "ebc51633c8807473",
              # 8 requests of 131,075 tokens: 2,152,513,536 bytes read (as ncu prints
              # them) for 2,152,120,864 algorithmic bytes; 3,049,728 bytes written by
              # 8 * 2 + 152 pieces
              "read_per_alg_byte": 2152513536 / 2152120864, "write_per_piece": 3049728 / 168}


# ------------------------------------------------------------ distributed

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(x: float, group=None) -> float:
    """Max of a float over all ranks (identity when not distributed)."""
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def reduce_sum(x: float) -> float:
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def shard_seed(base: int, rank: int) -> int:
    """Each rank serves its own shard of requests: same length distribution,
    its own data draw."""
    return base + 1000 * rank


# ------------------------------------------------------------ helpers

def algorithmic_bytes(w: wl.Workload, lens: np.ndarray, dtype: int, include_out=True) -> int:
    """Bytes the attention must move for one step: every valid cached K/V
    row, the per-page scales (e4m3), the page-table entries, Q, and O."""
    es = 1 if dtype == 0 else 2
    L = lens.astype(np.int64)
    pages = -(-L // w.page_size)
    kv = int((L * w.num_kv_heads * (w.head_dim_k + w.head_dim_v) * es).sum())
    scales = int((pages * w.num_kv_heads * 2 * 4).sum()) if dtype == 0 else 0
    pt = int((pages * 4).sum())
    q = w.B * w.q_tokens * w.num_q_heads * w.head_dim_k * 2
    o = w.B * w.q_tokens * w.num_q_heads * w.head_dim_v * 2 if include_out else 0
    return kv + scales + pt + q + o


def smi_index(local: int) -> str:
    """nvidia-smi id of this process's GPU (nvidia-smi ignores CUDA_VISIBLE_DEVICES)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if local < len(ids):
            return ids[local]
    return str(local)


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled through NVML
    (libnvidia-ml, the library nvidia-smi reads) every ~1 ms while a timed
    region runs: the decode steps last milliseconds, too short for
    nvidia-smi's 100 ms loop.  Read-only: no clock or setting is changed."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_id: str, period_s: float = 0.001):
        import ctypes
        import threading

        self.samples, self.masks, self.ok = [], [], False
        self.max_mhz = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            h = ctypes.c_void_p()
            if gpu_id.startswith("GPU-"):
                rc = lib.nvmlDeviceGetHandleByUUID(gpu_id.encode(), ctypes.byref(h))
            else:
                rc = lib.nvmlDeviceGetHandleByIndex_v2(int(gpu_id), ctypes.byref(h))
            if rc != 0:
                raise OSError(f"nvml handle rc={rc}")
            self.lib, self.h = lib, h
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # NVML_CLOCK_SM
                self.max_mhz = float(mx.value)
            reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.reasons_fn = reasons_fn
            self.ok = True
        except Exception as e:  # noqa: BLE001
            self.err = str(e)
            return
        self.stop_flag = False
        self.period = period_s
        self.t = threading.Thread(target=self._loop, daemon=True)
        self.t.start()

    def _loop(self):
        import ctypes

        c = ctypes.c_uint()
        m = ctypes.c_ulonglong()
        while not self.stop_flag:
            if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c)) == 0:
                self.samples.append(float(c.value))
            if self.reasons_fn(self.h, ctypes.byref(m)) == 0:
                self.masks.append(int(m.value))
            time.sleep(self.period)

    def stop(self) -> dict:
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None,
                    "reasons": [f"nvml unavailable: {getattr(self, 'err', '')}"]}
        self.stop_flag = True
        self.t.join(timeout=2)
        reasons = set()
        for m in self.masks:
            for bit, name in self.REASONS.items():
                if m & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "samples": len(self.samples),
                "reasons": sorted(reasons), "source": "nvml, ~1 ms period"}


# ------------------------------------------------------------ GPU arm

class Arm:
    """One pool (e4m3 or bf16) filled with the workload, ready to step."""

    def __init__(self, w: wl.Workload, dtype: int, device, total_steps: int, scale_mode=0):
        import paged_fp8_kv_append_gb300 as kv

        self.kv, self.w, self.dtype, self.device = kv, w, dtype, device
        self.pool = kv.KVPool(w.num_pages, w.page_size, w.num_kv_heads, w.head_dim_k,
                              w.head_dim_v, dtype=dtype, layout=w.layout, device=device,
                              tags=wl.initial_tags(w), free_list=wl.free_list(w),
                              scale_mode=scale_mode)
        B, mp = w.B, w.max_pages
        self.pt = torch.full((B, mp), -1, dtype=torch.int32, device=device)
        self.et = torch.zeros((B, mp), dtype=torch.int32, device=device)
        self.sl = torch.zeros(B, dtype=torch.int32, device=device)
        self.mask = torch.zeros(B, dtype=torch.uint8, device=device)
        self.out = torch.zeros((B, w.q_tokens, w.num_q_heads, w.head_dim_v), dtype=torch.bfloat16,
                               device=device)
        self.ws = torch.empty(self.pool.workspace_size(B, w.num_q_heads, w.q_tokens),
                              dtype=torch.uint8, device=device)
        self.ones = torch.arange(B + 1, dtype=torch.int32, device=device)  # 1 row per request
        # bulk fill: every request's first L_r - 1 tokens, a few requests per call
        lens0 = w.lens.astype(np.int64) - 1
        for r0 in range(0, B, 4):
            rs = list(range(r0, min(B, r0 + 4)))
            counts = np.zeros(B, np.int64)
            ks, vs = [], []
            for r in rs:
                k, v = wl.kv_rows(w, r, 0, int(lens0[r]), device=device)
                ks.append(k)
                vs.append(v)
                counts[r] = lens0[r]
            ind = torch.from_numpy(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32))
            self.pool.append(B, torch.cat(ks), torch.cat(vs), ind.to(device), int(counts.max()),
                             self.pt, self.et, self.sl)
            del ks, vs
        torch.cuda.synchronize()
        if self.pool.error() != 0:
            raise RuntimeError(f"fill failed: {kv.kv_status_string(self.pool.error())}")
        self.lens = w.lens.astype(np.int64).copy()  # length during the next step
        self.k_steps, self.v_steps, self.q_steps = [], [], []
        for s in range(total_steps):
            k, v = wl.step_rows(w, s, device=device)
            self.k_steps.append(k)
            self.v_steps.append(v)
            self.q_steps.append(wl.queries(w, device=device, step=s))
        self.step_no = 0

    def step(self, ev=None, launches=None, B=None):
        """append 1 token/request -> verify -> split -> combine, on the current
        stream, for the first B requests (all by default: the C ABI reads only
        the first B rows of every per-request array)."""
        kv, w, s = self.kv, self.w, self.step_no
        B = w.B if B is None else B
        h = self.pool.handle
        if ev is not None:
            ev[0].record()
        self.pool.append(B, self.k_steps[s], self.v_steps[s], self.ones, 1, self.pt, self.et,
                         self.sl)
        n = kv.kv_last_launch_count(h)
        if ev is not None:
            ev[1].record()
        self.pool.verify(B, self.pt, self.et, self.sl, self.mask)
        n += kv.kv_last_launch_count(h)
        if ev is not None:
            ev[2].record()
        kv.paged_decode_attn_split(h, B, w.num_q_heads, w.q_tokens, self.q_steps[s], self.pt,
                                   self.sl, self.mask, w.sm_scale, self.ws)
        n += kv.kv_last_launch_count(h)
        if ev is not None and ev[3] is not None:
            ev[3].record()
        kv.paged_decode_attn_combine(h, B, w.num_q_heads, w.q_tokens, self.mask, self.out, self.ws)
        n += kv.kv_last_launch_count(h)
        if ev is not None:
            ev[4].record()
        if launches is not None:
            launches.append(n)
        self.step_no += 1
        self.lens[:B] += 1

    def first_step_output(self, rs) -> dict:
        """Run the arm's first decode step (step rows 0, queries of step 0) and
        return the output rows of requests rs as bf16 bit patterns (host):
        the CPU-baseline leg replays the same step in the oracle."""
        assert self.step_no == 0
        self.out.fill_(7.0)
        self.step()
        torch.cuda.synchronize()
        if self.pool.error() != 0:
            raise RuntimeError(f"first step: {self.kv.kv_status_string(self.pool.error())}")
        return {int(r): wl.bits_u16(self.out[int(r)]) for r in rs}

    def run(self, steps: int, warmup: int, B=None, sync_ranks=True, split_event=True):
        """Eager steps, each call bracketed by CUDA events.  Returns (total ms,
        per-step ms [append, verify, split, combine], lengths, launches).
        split_event=False leaves out the event between the split and the
        combine (an event there keeps the combine's launch from overlapping
        the split's tail): column 2 is then the whole attention call and
        column 3 is zero."""
        B = self.w.B if B is None else B
        for _ in range(warmup):
            self.step(B=B)
        torch.cuda.synchronize()
        if sync_ranks:
            barrier()
        lens_timed = [self.lens[:B] + i for i in range(steps)]
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
        if not split_event:
            for e in evs:
                e[3] = None
        launches = []
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record()
        for i in range(steps):
            self.step(evs[i], launches, B=B)
        t1.record()
        torch.cuda.synchronize()
        total_ms = t0.elapsed_time(t1)
        if split_event:
            per = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(4)] for e in evs])
        else:
            per = np.array([[e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2]),
                             e[2].elapsed_time(e[4]), 0.0] for e in evs])
        err = self.pool.error()
        if err != 0:
            info = int(self.pool.ctl[3].item())
            raise RuntimeError(f"device error during timing: {self.kv.kv_status_string(err)} "
                               f"(wait info cta={info >> 12} warp={(info >> 7) & 31} "
                               f"barrier={(info >> 6) & 1} stage={info & 63}; dtype={self.dtype})")
        return total_ms, per, lens_timed, int(sum(launches))

    def run_graphs(self, steps: int, warmup: int, B=None, attention=True):
        """The next warmup + steps steps as CUDA graphs, one per step's inputs
        (a serving loop replays its decode step the same way), replayed in
        order, for the first B requests; each replay is a real decode step.
        attention=False leaves the split and combine out (append and tag
        check only).  Returns the timed steps' total ms."""
        kv, w, h = self.kv, self.w, self.pool.handle
        B = w.B if B is None else B

        def body(s):
            self.pool.append(B, self.k_steps[s], self.v_steps[s], self.ones, 1, self.pt,
                             self.et, self.sl)
            self.pool.verify(B, self.pt, self.et, self.sl, self.mask)
            if not attention:
                return
            kv.paged_decode_attn_split(h, B, w.num_q_heads, w.q_tokens, self.q_steps[s],
                                       self.pt, self.sl, self.mask, w.sm_scale, self.ws)
            kv.paged_decode_attn_combine(h, B, w.num_q_heads, w.q_tokens, self.mask, self.out,
                                         self.ws)

        s0, n = self.step_no, steps + warmup
        torch.cuda.synchronize()
        graphs = []
        for i in range(n):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                body(s0 + i)
            graphs.append(g)
        for i in range(warmup):
            graphs[i].replay()
        torch.cuda.synchronize()
        barrier()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for i in range(warmup, n):
            graphs[i].replay()
        t1.record()
        torch.cuda.synchronize()
        if self.pool.error() != 0:
            raise RuntimeError(f"graph steps: {self.kv.kv_status_string(self.pool.error())}")
        self.step_no += n
        self.lens[:B] += n
        del graphs
        return t0.elapsed_time(t1)

    def run_e2e(self, steps: int, warmup: int, graph: bool = True):
        """The next steps through host buffers and the one-call step API: per
        step, H2D copies of its new rows and queries from pinned host memory,
        kv_decode_step (tag check, append, attention), and D2H copies of the
        output and the abort mask into pinned memory, all inside the timed
        region.  graph: each step (copies included) is captured as a CUDA
        graph and the graphs are replayed in order, as a serving loop replays
        its step; otherwise every call is launched eagerly."""
        kv, w, B = self.kv, self.w, self.w.B
        n = steps + warmup
        s0 = self.step_no
        # one pinned staging buffer per step holding its K rows, V rows and
        # queries back to back (one H2D copy), and one device buffer holding
        # the output then the abort mask (one D2H copy)
        parts = [self.k_steps[0], self.v_steps[0], self.q_steps[0]]
        sizes = [t.numel() * 2 for t in parts]
        offs = np.concatenate([[0], np.cumsum(sizes)]).tolist()
        stage_h = []
        for i in range(n):
            buf = torch.empty(offs[-1], dtype=torch.uint8).pin_memory()
            for t, o, sz in zip((self.k_steps[s0 + i], self.v_steps[s0 + i],
                                 self.q_steps[s0 + i]), offs, sizes):
                buf[o:o + sz].copy_(t.cpu().contiguous().view(torch.uint8).reshape(-1))
            stage_h.append(buf)
        stage_d = torch.empty(offs[-1], dtype=torch.uint8, device=self.device)
        kd, vd, qd = (stage_d[o:o + sz].view(torch.bfloat16).view(t.shape)
                      for t, o, sz in zip(parts, offs, sizes))
        out_bytes = self.out.numel() * 2
        res_d = torch.empty(out_bytes + B, dtype=torch.uint8, device=self.device)
        out_d = res_d[:out_bytes].view(torch.bfloat16).view(self.out.shape)
        mask_d = res_d[out_bytes:]
        res_h = torch.empty(out_bytes + B, dtype=torch.uint8).pin_memory()
        ws = torch.empty(self.pool.step_workspace_size(B, w.num_q_heads, w.q_tokens),
                         dtype=torch.uint8, device=self.device)

        def one(i):
            stage_d.copy_(stage_h[i], non_blocking=True)
            self.pool.step(B, w.num_q_heads, w.q_tokens, None, kd, vd, self.ones, 1, self.pt,
                           self.et, self.sl, qd, w.sm_scale, out_d, mask_d, 0, ws)
            res_h.copy_(res_d, non_blocking=True)

        torch.cuda.synchronize()
        if graph:
            graphs = []
            for i in range(n):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    one(i)
                graphs.append(g)
            run = lambda i: graphs[i].replay()  # noqa: E731
        else:
            run = one
        for i in range(warmup):
            run(i)
        torch.cuda.synchronize()
        barrier()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for i in range(steps):
            run(warmup + i)
        t1.record()
        torch.cuda.synchronize()
        if self.pool.error() != 0:
            raise RuntimeError(f"e2e steps: {kv.kv_status_string(self.pool.error())}")
        if int(res_h[out_bytes:].sum()) != 0:
            raise RuntimeError("e2e steps: a request was aborted with every tag valid")
        self.step_no += n
        self.lens += n
        h2d, d2h = stage_d.numel(), res_d.numel()
        return t0.elapsed_time(t1), h2d, d2h


# ------------------------------------------------------------ bulk append

def bulk_append_line(w: wl.Workload, dtype: int, device, peak: float) -> dict:
    """One kv_append_quantize call that fills every request of a workload
    from empty (the prefill-to-decode handoff: bf16 rows in, e4m3 or bf16
    pages out), timed three times (median).  Algorithmic bytes: the bf16 rows read, the cache bytes
    written, and for e4m3 one fp32 scale per (page, kv head, K|V) written."""
    import paged_fp8_kv_append_gb300 as kv

    B, P = w.B, w.page_size
    pool = kv.KVPool(w.num_pages, P, w.num_kv_heads, w.head_dim_k, w.head_dim_v, dtype=dtype,
                     layout=w.layout, device=device, tags=wl.initial_tags(w),
                     free_list=wl.free_list(w))
    mp = w.max_pages
    pt = torch.full((B, mp), -1, dtype=torch.int32, device=device)
    et = torch.zeros((B, mp), dtype=torch.int32, device=device)
    sl = torch.zeros(B, dtype=torch.int32, device=device)
    lens = w.lens.astype(np.int64)
    ks, vs = [], []
    for r in range(B):
        k, v = wl.kv_rows(w, r, 0, int(lens[r]), device=device)
        ks.append(k)
        vs.append(v)
    k_all = torch.cat(ks)
    v_all = torch.cat(vs) if w.layout == 0 else None
    del ks, vs
    ind = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)).to(device)
    rel_ws = torch.empty(kv.kv_release_workspace_size(B), dtype=torch.uint8, device=device)
    # three fills of the same rows, the median reported: releasing every
    # request between fills hands the same pages back in the order they were
    # popped, so each fill writes the same pages
    times = []
    for rep in range(3):
        if rep > 0:
            pool.release(B, pt, et, sl, None, rel_ws)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        torch.cuda._sleep(1_000_000)
        e0.record()
        pool.append(B, k_all, v_all, ind, int(lens.max()), pt, et, sl)
        e1.record()
        torch.cuda.synchronize()
        if pool.error() != 0:
            raise RuntimeError(f"bulk append: {kv.kv_status_string(pool.error())}")
        times.append(e0.elapsed_time(e1))
    ms = float(np.median(times))
    rows = int(lens.sum())
    width = w.num_kv_heads * (w.head_dim_k + (w.head_dim_v if w.layout == 0 else 0))
    pages = int((-(-lens // P)).sum())
    out_b = rows * width * (1 if dtype == 0 else 2)
    scales = pages * (w.num_kv_heads * 2 if w.layout == 0 else 1) * 4 if dtype == 0 else 0
    byt = rows * width * 2 + out_b + scales
    del pool, k_all, v_all
    torch.cuda.empty_cache()
    return {"workload": w.name, "cache": "e4m3" if dtype == 0 else "bf16", "rows": rows,
            "ms": ms, "rows_per_s": rows / (ms / 1e3), "gbs": byt / (ms * 1e6),
            "pct_of_measured": 100.0 * byt / (ms * 1e6) / peak, "bytes": byt}


def handoff_line(w: wl.Workload, device, peak: float) -> dict:
    """kv_append_from_pool of every request of a workload: its rows read from
    a bf16 pool through that pool's page table into an empty e4m3 pool (the
    prefill-to-decode handoff without a gather copy), timed three times
    (median).  Algorithmic bytes: the bf16 rows read, the codes and one fp32
    scale per (page, kv head, K|V) written, the source page ids read and the
    destination page-table and expected-tag entries written."""
    import paged_fp8_kv_append_gb300 as kv

    B, P, mp = w.B, w.page_size, w.max_pages
    lens = w.lens.astype(np.int64)
    mk = lambda dt: kv.KVPool(w.num_pages, P, w.num_kv_heads, w.head_dim_k,  # noqa: E731
                              w.head_dim_v, dtype=dt, layout=w.layout, device=device,
                              tags=wl.initial_tags(w), free_list=wl.free_list(w))
    tabs = lambda: (torch.full((B, mp), -1, dtype=torch.int32, device=device),  # noqa: E731
                    torch.zeros((B, mp), dtype=torch.int32, device=device),
                    torch.zeros(B, dtype=torch.int32, device=device))
    src, (spt, set_, ssl) = mk(kv.KV_DTYPE_BF16), tabs()
    ind = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)).to(device)
    for r0 in range(0, B, 8):  # the source filled a few requests per call
        counts = np.zeros(B, np.int64)
        ks, vs = [], []
        for r in range(r0, min(B, r0 + 8)):
            k, v = wl.kv_rows(w, r, 0, int(lens[r]), device=device)
            ks.append(k)
            vs.append(v)
            counts[r] = lens[r]
        ind = torch.from_numpy(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32))
        src.append(B, torch.cat(ks), torch.cat(vs) if w.layout == 0 else None, ind.to(device),
                   int(counts.max()), spt, set_, ssl)
        del ks, vs
    dst, (pt, et, sl) = mk(kv.KV_DTYPE_E4M3), tabs()
    rel_ws = torch.empty(kv.kv_release_workspace_size(B), dtype=torch.uint8, device=device)
    times = []
    for rep in range(3):
        if rep > 0:
            dst.release(B, pt, et, sl, None, rel_ws)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        torch.cuda._sleep(1_000_000)
        e0.record()
        dst.append_from_pool(B, src, spt, ssl, pt, et, sl)
        e1.record()
        torch.cuda.synchronize()
        if dst.error() != 0 or src.error() != 0:
            raise RuntimeError(f"handoff: {kv.kv_status_string(dst.error() or src.error())}")
        times.append(e0.elapsed_time(e1))
    ms = float(np.median(times))
    rows = int(lens.sum())
    width = w.num_kv_heads * (w.head_dim_k + (w.head_dim_v if w.layout == 0 else 0))
    pages = int((-(-lens // P)).sum())
    scales = pages * (w.num_kv_heads * 2 if w.layout == 0 else 1) * 4
    byt = rows * width * 2 + rows * width + scales + pages * (4 + 8)
    del src, dst
    torch.cuda.empty_cache()
    return {"workload": w.name, "cache": "bf16 pool -> e4m3 pool", "rows": rows, "ms": ms,
            "rows_per_s": rows / (ms / 1e3), "gbs": byt / (ms * 1e6),
            "pct_of_measured": 100.0 * byt / (ms * 1e6) / peak, "bytes": byt}


# ------------------------------------------------------------ re-quantising scale mode

def dequant_rel_error(pool, pt, lens, src_k, P: int) -> float:
    """Worst per-row relative error of the dequantised K rows of the last
    appended token of every request against the bf16 rows appended:
    max |deq - x| / max |x| over each (request, kv head) row."""
    import paged_fp8_kv_append_gb300 as kv  # noqa: F401

    worst = 0.0
    for r in range(len(lens)):
        pos = int(lens[r]) - 1
        p = int(pt[r, pos // P].item())
        codes = pool.k_cache[p, :, pos % P, :]                       # [Hkv][D] uint8
        deq = codes.view(torch.float8_e4m3fn).float() * pool.k_scale[p][:, None]
        x = src_k[r].float()                                          # [Hkv][D]
        err = (deq - x).abs().amax(dim=1) / x.abs().amax(dim=1).clamp_min(1e-30)
        worst = max(worst, float(err.max()))
    return worst


def requant_lines(device, steps: int, warmup: int, w: wl.Workload) -> dict:
    """KV_SCALE_REQUANTIZE: the decode step's append with it on the GQA batch,
    and its effect on a stream whose single-token rows grow 1.35x per step
    (frozen scales saturate the larger rows; re-quantised ones keep them)."""
    arm = Arm(w, 0, device, steps + warmup, scale_mode=1)
    _, per, _, _ = arm.run(steps, warmup, sync_ranks=False)
    out = {"append_us_requantize": float(per[:, 0].mean() * 1e3)}
    del arm
    torch.cuda.empty_cache()
    # accuracy on a growing stream: 32 requests of 20 rows, then 16 growing steps
    import paged_fp8_kv_append_gb300 as kv

    lens = np.full(32, 20, np.int32)
    sw = wl.Workload("growth", 20267, lens, 64, 8, 128, 128, 16, 1, 0, 32 * 4 + 64,
                     float(np.float32(1 / np.sqrt(128))), steps=20)
    for mode in (0, 1):
        pool = kv.KVPool(sw.num_pages, 16, 8, 128, 128, dtype=0, layout=0, device=device,
                         tags=wl.initial_tags(sw), free_list=wl.free_list(sw), scale_mode=mode)
        B, mp = sw.B, sw.max_pages
        pt = torch.full((B, mp), -1, dtype=torch.int32, device=device)
        et = torch.zeros((B, mp), dtype=torch.int32, device=device)
        sl = torch.zeros(B, dtype=torch.int32, device=device)
        k0 = torch.cat([wl.kv_rows(sw, r, 0, 20, device=device)[0] for r in range(B)])
        v0 = torch.cat([wl.kv_rows(sw, r, 0, 20, device=device)[1] for r in range(B)])
        ind = torch.arange(0, 21 * B, 20, dtype=torch.int32, device=device)[:B + 1]
        pool.append(B, k0, v0, ind, 20, pt, et, sl)
        ones = torch.arange(B + 1, dtype=torch.int32, device=device)
        worst = 0.0
        for st in range(16):
            k, v = wl.step_rows(sw, st, device=device)
            g = 1.35 ** (st + 1)
            k, v = (k.float() * g).to(torch.bfloat16), (v.float() * g).to(torch.bfloat16)
            pool.append(B, k, v, ones, 1, pt, et, sl)
            worst = max(worst, dequant_rel_error(pool, pt, sl.cpu().numpy(), k, 16))
        out[f"stream_max_rel_error_{'requantize' if mode else 'frozen'}"] = worst
        del pool
    out["stream"] = ("32 requests of 20 rows, then 16 single-token steps whose rows grow 1.35x "
                     "per step; worst per-row relative error of the newest K row, dequantised")
    return out


# ------------------------------------------------------------ continuous batching

def _churn(device, steps: int, warmup: int, driver: bool) -> dict:
    """One churn run (see churn_line).  driver: every step is one
    kv_decode_step call (leavers released, joiners' prompts and everyone
    else's new row appended together, tag check, attention, aborted requests
    removed); otherwise the same work as separate calls (release, the
    joiners' bulk append, then a decode step: append, verify, attention)."""
    import math as _m

    rng = np.random.default_rng(20268)
    S = 128

    def prompt_lens(n):
        return np.clip(np.round(rng.lognormal(_m.log(4096), 1.0, n)), 512, 32768).astype(np.int32)

    lens = prompt_lens(S)
    n_steps = steps + warmup
    w = wl.Workload("churn", 20268, lens, 64, 8, 128, 128, 16, 1, 0,
                    int((-(-lens.astype(np.int64) // 16)).sum() * 2) + 4096,
                    float(np.float32(1 / np.sqrt(128))), steps=32768 + n_steps)
    arm = Arm(w, 0, device, n_steps)
    kv = arm.kv
    rel_ws = torch.empty(kv.kv_release_workspace_size(S), dtype=torch.uint8, device=device)
    step_ws = torch.empty(arm.pool.step_workspace_size(S, w.num_q_heads, w.q_tokens),
                          dtype=torch.uint8, device=device)
    phase = {"release": [], "join": [], "step": []}
    totals, rows_per_step = [], []
    for it in range(n_steps):
        leave = rng.choice(S, 3, replace=False)
        mask = np.zeros(S, np.uint8)
        mask[leave] = 1
        new = prompt_lens(3)
        m_d = torch.from_numpy(mask).to(device)
        prompts = {}
        for r, n in zip(leave, new):
            prompts[int(r)] = wl.kv_rows(w, int(r), 0, int(n), device=device, tag=1000 + it)
        if driver:
            counts = np.ones(S, np.int64)
            ks, vs = [], []
            for r in range(S):
                if r in prompts:  # the prompt, then its first decode row
                    counts[r] = prompts[r][0].shape[0] + 1
                    ks.append(prompts[r][0])
                    vs.append(prompts[r][1])
                ks.append(arm.k_steps[it][r:r + 1])
                vs.append(arm.v_steps[it][r:r + 1])
            k_new, v_new = torch.cat(ks), torch.cat(vs)
            ind = torch.from_numpy(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)).to(device)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            torch.cuda.synchronize()
            torch.cuda._sleep(1_000_000)
            ev[0].record()
            arm.pool.step(S, w.num_q_heads, w.q_tokens, m_d, k_new, v_new, ind,
                          int(counts.max()), arm.pt, arm.et, arm.sl, arm.q_steps[it], w.sm_scale,
                          arm.out, arm.mask, kv.KV_STEP_REMOVE_ABORTED, step_ws)
            ev[1].record()
            torch.cuda.synchronize()
            if it >= warmup:
                totals.append(ev[0].elapsed_time(ev[1]))
                rows_per_step.append(int(counts.sum()))
        else:
            counts = np.zeros(S, np.int64)
            counts[leave] = new
            k_new = torch.cat([prompts[int(r)][0] for r in leave])
            v_new = torch.cat([prompts[int(r)][1] for r in leave])
            ind = torch.from_numpy(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)).to(device)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            torch.cuda.synchronize()
            torch.cuda._sleep(1_000_000)
            ev[0].record()
            arm.pool.release(S, arm.pt, arm.et, arm.sl, m_d, rel_ws)
            ev[1].record()
            arm.pool.append(S, k_new, v_new, ind, int(new.max()), arm.pt, arm.et, arm.sl)
            ev[2].record()
            arm.step()
            ev[3].record()
            torch.cuda.synchronize()
            if it >= warmup:
                for k_, (a, b) in zip(("release", "join", "step"), ((0, 1), (1, 2), (2, 3))):
                    phase[k_].append(ev[a].elapsed_time(ev[b]))
                totals.append(ev[0].elapsed_time(ev[3]))
        if arm.pool.error() != 0:
            raise RuntimeError(f"churn: {kv.kv_status_string(arm.pool.error())}")
        if driver and int(arm.mask.sum().item()) != 0:
            raise RuntimeError("churn: a request was aborted with every tag valid")
    del arm
    torch.cuda.empty_cache()
    t = float(np.sum(totals))
    res = {"decode_tokens_per_s": S * len(totals) / (t / 1e3),
           "us_per_step": float(np.mean(totals) * 1e3)}
    if driver:
        res["rows_appended_per_step"] = float(np.mean(rows_per_step))
    else:
        res["us"] = {k_: float(np.mean(v) * 1e3) for k_, v in phase.items()}
    return res


def churn_line(device, steps: int, warmup: int) -> dict:
    """Continuous batching over 128 request slots (64 q / 8 kv heads, head dim
    128, page 16, e4m3; prompts lognormal, median 4k tokens, in [512, 32k]).
    Every step, 3 requests finish and release their pages, 3 new ones join
    the freed slots with their prompts, and every slot takes a decode step.
    Measured two ways on the same seeded workload: one kv_decode_step call
    per step, and the same work as separate calls (with its phase times)."""
    return {"workload": "churn: 128 request slots, 64 q / 8 kv heads, head dim 128, page 16, "
                        "e4m3; prompts lognormal (median 4k) in [512, 32k]; per step 3 leave "
                        "and 3 join with their prompts, then every slot decodes one token",
            "step_driver": _churn(device, steps, warmup, True),
            "separate_calls": _churn(device, steps, warmup, False)}


# ------------------------------------------------------------ wider query groups

def wide_group_line(device, steps: int, warmup: int, peak: float, B: int = 32,
                    dtype: int = 0, parity=None) -> dict:
    """The GQA batch's requests with 96 query heads on its 8 kv heads (the
    GLM-class group of 12): 12 query rows per kv head, each kv head's rows
    served by one 16-row consumer warp.  e4m3 (dtype 0) or bf16 (1); the step
    is append -> verify -> split -> combine as in the headline.  B < 32: the
    first B requests (small profiling captures)."""
    import dataclasses

    w = dataclasses.replace(wl.gqa_batch(steps=3 * (steps + warmup) + 2), num_q_heads=96)
    if B != w.B:
        w = wl.subset(w, B)
    arm = Arm(w, dtype, device, 1 + 3 * (steps + warmup))
    if parity is not None:
        r = int(np.argmax(w.lens))
        parity.append({"name": f"wide96_{'e4m3' if dtype == 0 else 'bf16'}", "w": w,
                       "dtype": dtype, "pairs": [(r, 6)], "outs": arm.first_step_output([r])})
    line = step_line(w, arm, dtype, steps, warmup)
    line["pct_of_measured"] = 100.0 * line["attn_gbs"] / peak
    line["workload"] = (f"gqa_batch with 96 q / 8 kv heads (12 query rows per kv head): {w.B} "
                        "requests, contexts U[4096, 32768], head dim 128, page 16, "
                        + ("e4m3" if dtype == 0 else "bf16"))
    del arm
    torch.cuda.empty_cache()
    return line


# ------------------------------------------------------------ verify overhead

def overhead_tokens(replays: int) -> int:
    """Tokens one graph_overhead call appends to each measured request (at
    most: a short step takes five times the rounds)."""
    return 3 * (5 + 5 * replays) + 1


def graph_overhead(arm: "Arm", replays: int, B=None) -> dict:
    """Cost of the page-tag check inside a whole step: two CUDA graphs of the
    same step structure, append -> verify -> split -> combine and append ->
    split -> combine with no abort mask, replayed alternately; overhead =
    median(with) / median(without) - 1.  All tags are valid, so both attend
    exactly the same requests.  Each replay is a real decode step (one more
    token per request)."""
    kv, w, h = arm.kv, arm.w, arm.pool.handle
    B = w.B if B is None else B
    k0, v0, q0 = arm.k_steps[0], arm.v_steps[0], arm.q_steps[0]

    def body(check: str):
        arm.pool.append(B, k0, v0, arm.ones, 1, arm.pt, arm.et, arm.sl)
        if check == "fused":  # the tag check inside the page reads
            kv.paged_decode_attn_checked(h, B, w.num_q_heads, w.q_tokens, q0, arm.pt, arm.et,
                                         arm.sl, w.sm_scale, arm.out, arm.mask, arm.ws)
            return
        mask = None
        if check == "separate":
            arm.pool.verify(B, arm.pt, arm.et, arm.sl, arm.mask)
            mask = arm.mask
        kv.paged_decode_attn_split(h, B, w.num_q_heads, w.q_tokens, q0, arm.pt, arm.sl, mask,
                                   w.sm_scale, arm.ws)
        kv.paged_decode_attn_combine(h, B, w.num_q_heads, w.q_tokens, mask, arm.out, arm.ws)

    modes = ("separate", "none", "fused")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for m in modes:
            body(m)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graphs = {m: torch.cuda.CUDAGraph() for m in modes}
    for m in modes:
        with torch.cuda.graph(graphs[m]):
            body(m)
    for _ in range(3):
        for m in modes:
            graphs[m].replay()
    torch.cuda.synchronize()
    # each round replays the three graphs in a rotated order (no mode always
    # runs first after the round's start); short steps take more rounds
    for m in modes:
        graphs[m].replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    graphs["none"].replay()
    e1.record()
    torch.cuda.synchronize()
    if e0.elapsed_time(e1) < 0.5:
        replays *= 5
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(replays)]
    order = [[modes[(i + j) % 3] for j in range(3)] for i in range(replays)]
    for i in range(replays):
        ev[i][0].record()
        for j, m in enumerate(order[i]):
            graphs[m].replay()
            ev[i][j + 1].record()
    torch.cuda.synchronize()
    if arm.pool.error() != 0:
        raise RuntimeError(f"verify overhead: device error {kv.kv_status_string(arm.pool.error())}")
    if int(arm.mask[:B].sum().item()) != 0:
        raise RuntimeError("verify overhead: a request was aborted with every tag valid")
    # every run of the body appended one token
    arm.lens[:B] += len(modes) * (1 + 3 + 1 + replays) + 1
    t = {m: [] for m in modes}
    for i in range(replays):
        for j, m in enumerate(order[i]):
            t[m].append(ev[i][j].elapsed_time(ev[i][j + 1]))
    med = {m: statistics.median(t[m]) for m in modes}
    del graphs
    return {"workload": w.name, "requests": B, "replays": replays,
            "ms_with_verify": med["separate"], "ms_without_verify": med["none"],
            "ms_fused_check": med["fused"],
            "verify_overhead_pct": 100.0 * (med["separate"] / med["none"] - 1.0),
            "fused_overhead_pct": 100.0 * (med["fused"] / med["none"] - 1.0),
            "mean_overhead_pct": 100.0 * (sum(t["separate"]) / sum(t["none"]) - 1.0)}


def step_line(w: wl.Workload, arm: "Arm", dtype: int, steps: int, warmup: int, B=None,
              aborted=()) -> dict:
    """tokens/s of the whole step (non-aborted requests / summed kernel time)
    and GB/s of split + combine over the algorithmic bytes of the requests
    attended, for the first B requests of an Arm."""
    B = w.B if B is None else B
    total_ms, per, lens_timed, _ = arm.run(steps, warmup, B=B, sync_ranks=False,
                                           split_event=False)
    graph_ms = arm.run_graphs(steps, warmup, B=B)
    graph_noattn_ms = arm.run_graphs(steps, warmup, B=B, attention=False)
    keep = np.array([r not in set(aborted) for r in range(B)])
    sub = wl.subset(w, B)
    byt = []
    for L in lens_timed:
        Lk = np.where(keep, L, 0)
        b = algorithmic_bytes(sub, Lk, dtype)
        # Q and O only for the requests attended
        b -= (B - int(keep.sum())) * sub.q_tokens * sub.num_q_heads * (sub.head_dim_k +
                                                                       sub.head_dim_v) * 2
        byt.append(b)
    attn_ms = per[:, 2]
    gbs = float(np.mean([b / (t * 1e6) for b, t in zip(byt, attn_ms)]))
    # the attention's share of a CUDA-graph step: the step with it minus the
    # same step without it (append and tag check only)
    attn_graph_us = (graph_ms - graph_noattn_ms) / steps * 1e3
    gbs_graph = float(np.mean(byt)) / (attn_graph_us * 1e3)
    return {"requests": B, "attended": int(keep.sum()),
            "attn_us_graph": attn_graph_us, "attn_gbs_graph": gbs_graph,
            "tokens_per_s": int(keep.sum()) * w.q_tokens * steps / (graph_ms / 1e3),
            "ms_per_step": graph_ms / steps, "eager_ms_per_step": total_ms / steps,
            "attn_us": float(attn_ms.mean() * 1e3),
            "attn_gbs": gbs, "pct_of_8000": 100.0 * gbs / NOMINAL_HBM_GBS,
            "kernel_us": {k: float(per[:, i].mean() * 1e3)
                          for i, k in enumerate(("append", "verify", "attention"))},
            "timing": "tokens/s: each step a CUDA graph replay; attention: CUDA events around "
                      "the split + combine calls of eager steps; attn_us_graph: CUDA-graph "
                      "step time with the attention minus without it"}


def sweep_lines(w: wl.Workload, arm: "Arm", dtype: int, steps: int, warmup: int, peak: float,
                points) -> list:
    """Step lines (tokens/s, attention GB/s) for the first B requests of a
    filled 131,072-token pool, for each B in points."""
    out = []
    for B in points:
        line = step_line(w, arm, dtype, steps, warmup, B=B)
        line["pct_of_measured"] = 100.0 * line["attn_gbs"] / peak
        out.append(line)
    return out


def release_lines(arm: "Arm") -> list:
    """kv_release_pages on a filled pool: a seeded 10% of the requests, then
    all the others.  Algorithmic bytes: 16 per page (its id read, written to
    the free list, its page-table entry and expected tag cleared)."""
    w, B = arm.w, arm.w.B
    P = w.page_size
    sel = np.zeros(B, np.uint8)
    sel[np.random.default_rng(w.seed + 7).choice(B, max(1, B // 10), replace=False)] = 1
    ws = torch.empty(arm.kv.kv_release_workspace_size(B), dtype=torch.uint8, device=arm.device)
    # an empty release first: loads the kernels, changes nothing
    arm.pool.release(B, arm.pt, arm.et, arm.sl, torch.zeros(B, dtype=torch.uint8,
                                                            device=arm.device), ws)
    out = []
    for name, mask in (("10% of requests", sel), ("the other 90%", 1 - sel)):
        L = arm.sl.cpu().numpy().astype(np.int64)
        pages = int((-(-L // P) * mask).sum())
        m_d = torch.from_numpy(mask).to(arm.device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        # keep the GPU busy while the host enqueues, so the events time the
        # kernels and not the launch calls
        torch.cuda._sleep(1_000_000)
        e0.record()
        arm.pool.release(B, arm.pt, arm.et, arm.sl, m_d, ws)
        e1.record()
        torch.cuda.synchronize()
        if arm.pool.error() != 0:
            raise RuntimeError(f"release: {arm.kv.kv_status_string(arm.pool.error())}")
        us = e0.elapsed_time(e1) * 1e3
        out.append({"released": name, "requests": int(mask.sum()), "pages": pages, "us": us,
                    "gbs": 16.0 * pages / (us * 1e3)})
    return out


def skewed_lines(device, replays: int, steps: int, warmup: int, peak: float, parity=None):
    """The skewed long-context stress workload (256 requests, lognormal
    contexts, median 16k, up to 256k; 32 q / 4 kv heads, e4m3, page 16; about
    428k pages checked per step): the verify overhead with every tag valid,
    then the full step with its seeded stale tags (those requests abort)."""
    w = wl.skewed(steps=overhead_tokens(replays) + 3 * (steps + warmup) + 8)
    stale = list(w.stale)
    w.stale = []  # every tag valid: both graphs attend the same requests
    arm = Arm(w, 0, device, 1 + 3 * (steps + warmup))
    if parity is not None:  # a seeded live request, all tags valid at this step
        live = [r for r in range(w.B) if r not in stale and w.lens[r] <= 65536]
        r = int(np.random.default_rng(w.seed + 11).choice(live))
        parity.append({"name": "skewed_e4m3", "w": w, "dtype": 0, "pairs": [(r, 3)],
                       "outs": arm.first_step_output([r])})
    over = graph_overhead(arm, replays)
    over["workload"] = ("skewed: 256 requests, lognormal contexts (median 16k) in [1, 256k], "
                        "32 q / 4 kv heads, head dim 128, page 16, e4m3; all tags valid")
    over["pages_checked_per_step"] = int((-(-(w.lens.astype(np.int64)) // 16)).sum())
    # the step as the workload defines it: one seeded stale tag in 1% of requests
    w.stale = stale
    et = arm.et.cpu().numpy().view(np.uint32).copy()
    for r, j in wl.stale_slots(w):
        et[r, j] = np.uint32(et[r, j]) - np.uint32(1)
    arm.et.copy_(torch.from_numpy(et.view(np.int32)))
    arm.step_no = 1
    line = step_line(w, arm, 0, steps, warmup, aborted=stale)
    if not np.array_equal(np.flatnonzero(arm.mask.cpu().numpy()), np.array(sorted(stale))):
        raise RuntimeError("skewed step: abort mask differs from the stale requests")
    line["pct_of_measured"] = 100.0 * line["attn_gbs"] / peak
    line["aborted"] = sorted(stale)
    line["workload"] = ("skewed: 256 requests, lognormal contexts (median 16k) in [1, 256k], "
                        "32 q / 4 kv heads, head dim 128, page 16, e4m3; 3 stale requests abort")
    line["release"] = release_lines(arm)
    del arm
    torch.cuda.empty_cache()
    return over, line


# ------------------------------------------------------------ latent verify

def latent_flops(w: wl.Workload, lens: np.ndarray) -> float:
    """Algorithmic flops of one latent attention call: every query row t of
    request r sees L_r - T + t + 1 positions, 2*(Dk + Dv) flops each."""
    T = w.q_tokens
    vis = sum(int(L) - T + t + 1 for L in lens for t in range(T))
    return 2.0 * vis * w.num_q_heads * (w.head_dim_k + w.head_dim_v)


def latent_bench(steps: int, warmup: int, device, peaks: dict, B: int = 64) -> dict:
    """One decode step of the latent speculative-verify workload (64 requests,
    lognormal contexts 8k..64k, 128 heads x 4 draft tokens on one 576-wide
    e4m3 row per token): append the 4 draft rows of every request, tag check,
    attention (tcgen05 path) + combine."""
    import paged_fp8_kv_append_gb300 as kv

    w = wl.latent_verify(B=B)
    T, B = w.q_tokens, w.B
    w.steps = T * (steps + warmup + 1)
    import math as _m

    need = int((-(-(w.lens.astype(np.int64) + w.steps) // 64)).sum())
    w.num_pages = int(_m.ceil(need * 1.1)) + 8
    pool = kv.KVPool(w.num_pages, 64, 1, 576, 512, dtype=0, layout=1, device=device,
                     tags=wl.initial_tags(w), free_list=wl.free_list(w))
    mp = w.max_pages
    pt = torch.full((B, mp), -1, dtype=torch.int32, device=device)
    et = torch.zeros((B, mp), dtype=torch.int32, device=device)
    sl = torch.zeros(B, dtype=torch.int32, device=device)
    lens0 = w.lens.astype(np.int64) - T
    for r0 in range(0, B, 8):
        counts = np.zeros(B, np.int64)
        ks = []
        for r in range(r0, min(B, r0 + 8)):
            counts[r] = lens0[r]
            ks.append(wl.kv_rows(w, r, 0, int(lens0[r]), device=device)[0])
        ind = torch.from_numpy(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32))
        pool.append(B, torch.cat(ks), None, ind.to(device), int(counts.max()), pt, et, sl)
        del ks
    mask = torch.zeros(B, dtype=torch.uint8, device=device)
    out = torch.zeros((B, T, w.num_q_heads, 512), dtype=torch.bfloat16, device=device)
    ws = torch.empty(pool.workspace_size(B, w.num_q_heads, T), dtype=torch.uint8, device=device)
    ind_t = torch.arange(0, (B + 1) * T, T, dtype=torch.int32, device=device)
    g = torch.Generator(device=device)
    drafts, qs = [], []
    for s in range(steps + warmup):
        g.manual_seed(w.seed * 17 + s)
        drafts.append(torch.randn((B * T, 576), generator=g, device=device).to(torch.bfloat16))
        qs.append(wl.queries(w, device=device, step=s))
    lens = w.lens.astype(np.int64).copy()

    def step(s, ev=None):
        pool.append(B, drafts[s], None, ind_t, T, pt, et, sl)
        pool.verify(B, pt, et, sl, mask)
        if ev is not None:
            ev[0].record()
        pool.attn(B, w.num_q_heads, T, qs[s], pt, sl, mask, w.sm_scale, out, ws)
        if ev is not None:
            ev[1].record()

    for s in range(warmup):
        step(s)
    torch.cuda.synchronize()
    lens += T * warmup
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    flops = []
    for i in range(steps):
        step(warmup + i, evs[i])
        flops.append(latent_flops(w, lens + T * i))
    t1.record()
    torch.cuda.synchronize()
    if pool.error() != 0:
        raise RuntimeError(f"latent: device error {kv.kv_status_string(pool.error())}")
    total = t0.elapsed_time(t1)
    attn_ms = np.array([e[0].elapsed_time(e[1]) for e in evs])
    tf = float(np.mean([f / (t * 1e-3) / 1e12 for f, t in zip(flops, attn_ms)]))
    peak = float(peaks.get("bf16_tflops", 1900.0))
    kv_bytes = float((lens + T * steps // 2).sum() * 576 + B * T * 128 * (576 + 512) * 2)
    res = {"workload": f"latent_verify: {B} requests, lognormal contexts (median 16k) in "
                       "[8k, 64k], 128 heads x 4 draft tokens, one 576-wide e4m3 row per token "
                       "(V = first 512), page 64",
           "value": steps * B * T / (total / 1e3), "unit": "tokens/s",
           "ms_per_step": total / steps, "attn_ms": float(attn_ms.mean()),
           "attn_tflops": tf, "tensor_peak_tflops": peak, "tensor_frac": tf / peak,
           "peak_source": "measured bf16 dense (f16 operands run at the same rate)",
           "attn_gbs": kv_bytes / (attn_ms.mean() * 1e6)}
    del pool
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------ CPU oracle

TOL_ABS, TOL_REL = 2e-3, 1e-2  # attention tolerance: |o - r| <= abs + rel * |r|


def _bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
        torch.bfloat16).to(torch.float64).numpy()


def oracle_pair_step(w: wl.Workload, r: int, h: int, dtype: int, device):
    """The oracle's replay of the first decode step of request r of a GQA
    workload, for its kv head h only (a one-kv-head pool fed that head's
    rows, as the GPU arms feed all heads): the request's first L_r - 1 rows
    appended in one call (untimed), then the timed step -- the step's new row
    appended, the tag check, fp64 attention for the G query heads of kv head
    h.  Returns (seconds of the timed step, output [T][G][Dv])."""
    import oracle

    T, P = w.q_tokens, w.page_size
    G = w.num_q_heads // w.num_kv_heads
    L = int(w.lens[r])
    npg = -(-L // P) + 1
    ptab = np.full((1, npg), -1, np.int32)
    et = np.zeros((1, npg), np.uint32)
    sl = np.zeros(1, np.int32)
    n0 = L - T
    k, v = wl.kv_rows(w, r, 0, n0, device=device)
    pool = oracle.Pool(npg, P, 1, w.head_dim_k, w.head_dim_v, dtype=dtype)
    oracle.append(pool, wl.bits_u16(k[:, h:h + 1]), wl.bits_u16(v[:, h:h + 1]),
                  np.array([0, n0], np.int32), n0, ptab, et, sl)
    del k, v
    ks, vs = wl.step_rows(w, 0, device=device)
    krow, vrow = wl.bits_u16(ks[r:r + 1, h:h + 1]), wl.bits_u16(vs[r:r + 1, h:h + 1])
    q = wl.bits_u16(wl.queries(w, device=device)[r:r + 1, :, h * G:(h + 1) * G])
    t0 = time.perf_counter()
    oracle.append(pool, krow, vrow, np.array([0, T], np.int32), T, ptab, et, sl)
    mask = oracle.verify(pool.num_pages, P, pool.tags, ptab, et, sl)
    ref, written = oracle.attn(pool, q, ptab, sl, mask, w.sm_scale, G, T)
    sec = time.perf_counter() - t0
    if not written[0]:
        raise RuntimeError(f"oracle: request {r} of {w.name} aborted with every tag valid")
    return sec, ref[0]


def cpu_baseline_leg(samples: list, device, budget_s: float) -> tuple:
    """The CPU oracle, as it stands, on one host core: it replays the first
    decode step of sampled (request, kv head) pairs of the timed workloads
    (the GPU's output rows of that step were kept) and compares them element
    by element.  The headline's pairs give the baseline's tokens/s (a pair is
    1/Hkv of a request's decode token); every pair gives a parity record.
    Samples after the first two stop once budget_s of timed oracle work is
    spent."""
    head_sec, head_tok, head_names = 0.0, 0.0, []
    parity, spent = {}, 0.0
    for i, smp in enumerate(samples):
        w, name = smp["w"], smp["name"]
        G = w.num_q_heads // w.num_kv_heads
        for r, h in smp["pairs"]:
            if i >= 2 and spent > budget_s:
                break
            sec, ref = oracle_pair_step(w, r, h, smp["dtype"], device)
            spent += sec
            got = _bf16_bits_to_f64(smp["outs"][r])[:, h * G:(h + 1) * G]
            err = np.abs(got - ref)
            ok = bool(np.all(err <= TOL_ABS + TOL_REL * np.abs(ref)))
            rel = float((err / np.maximum(np.abs(ref), 1e-30)).max())
            p = parity.setdefault(name, {"ok": True, "max_abs": 0.0, "max_rel": 0.0,
                                         "pairs": []})
            p["ok"] = p["ok"] and ok
            p["max_abs"] = max(p["max_abs"], float(err.max()))
            p["max_rel"] = max(p["max_rel"], rel)
            p["pairs"].append([int(r), int(h)])
            if smp.get("headline"):
                head_sec += sec
                head_tok += w.q_tokens / w.num_kv_heads
                head_names.append(f"r{r}/kv{h}(L={int(w.lens[r])})")
    return head_tok, head_sec, head_names, parity


def reference_arm(args):
    """--impl reference: the oracle, as it stands, on the headline workload
    (requests of 131,072 tokens; 64 q / 8 kv heads, head dim 128, page 16,
    e4m3), on one host core.  Each step is one decode step of one (request,
    kv head) pair -- its new row appended, the tag check, fp64 attention for
    the kv head's 8 query heads -- so a step is 1/8 of a request's decode
    token; the pair's earlier rows are appended once before the first step."""
    import oracle

    ws, rank, _ = dist_env()
    if rank != 0:
        return
    device = "cuda" if torch.cuda.is_available() else "cpu"
    w = wl.concurrency(64)
    r, h, L, P = 0, 0, int(w.lens[0]), w.page_size
    G = w.num_q_heads // w.num_kv_heads
    n = args.warmup + args.steps
    npg = -(-(L + n) // P) + 1
    pool = oracle.Pool(npg, P, 1, w.head_dim_k, w.head_dim_v, dtype=0)
    ptab = np.full((1, npg), -1, np.int32)
    et = np.zeros((1, npg), np.uint32)
    sl = np.zeros(1, np.int32)
    k, v = wl.kv_rows(w, r, 0, L - 1, device=device)
    oracle.append(pool, wl.bits_u16(k[:, h:h + 1]), wl.bits_u16(v[:, h:h + 1]),
                  np.array([0, L - 1], np.int32), L - 1, ptab, et, sl)
    del k, v
    per_step = []
    for i in range(n):
        ks, vs = wl.step_rows(w, i, device=device)
        q = wl.bits_u16(wl.queries(w, device=device, step=i)[r:r + 1, :, h * G:(h + 1) * G])
        krow, vrow = wl.bits_u16(ks[r:r + 1, h:h + 1]), wl.bits_u16(vs[r:r + 1, h:h + 1])
        t0 = time.perf_counter()
        oracle.append(pool, krow, vrow, np.array([0, 1], np.int32), 1, ptab, et, sl)
        mask = oracle.verify(pool.num_pages, P, pool.tags, ptab, et, sl)
        oracle.attn(pool, q, ptab, sl, mask, w.sm_scale, G, w.q_tokens)
        if i >= args.warmup:
            per_step.append(time.perf_counter() - t0)
    total = sum(per_step)
    value = args.steps * w.q_tokens / w.num_kv_heads / total
    sample = (f"{args.steps} decode steps of request 0 (131,072+ tokens), kv head 0 (8 query "
              "heads, 1/8 of a request's token each) of the 64 x 131,072 e4m3 workload, one per "
              "step, on one host core")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": HEADLINE_NAME, "batch_per_step": "1 (request, kv head) pair",
                   "note": "CPU oracle: each step is one (request, kv head) decode step (append "
                           "1 row, tag check, fp64 attention of 8 query heads)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ------------------------------------------------------------ main

HEADLINE_NAME = ("concurrency 64 x 131072: 64 requests of 131,072 tokens, 64 q / 8 kv heads, "
                 "head dim 128, page 16, e4m3")


def _peaks() -> dict:
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:  # noqa: BLE001
        return {}


def _pt(line: dict, peak: float) -> dict:
    """Compact summary of a step line: tokens/s, attention GB/s (eager call)
    and its fraction of the measured copy bandwidth and of 8 TB/s, and the
    same from the attention's share of a CUDA-graph step (`*_graph`)."""
    d = {"tok_s": round(line["tokens_per_s"], 1), "gbs": round(line["attn_gbs"], 1),
         "frac": round(line["attn_gbs"] / peak, 4),
         "frac_8000": round(line["attn_gbs"] / NOMINAL_HBM_GBS, 4),
         "attn_us": round(line["attn_us"], 2)}
    if "attn_gbs_graph" in line:
        d["frac_graph"] = round(line["attn_gbs_graph"] / peak, 4)
        d["attn_us_graph"] = round(line["attn_us_graph"], 2)
    return d


def split_traffic(alg_bytes: float, pieces: int):
    """DRAM bytes of one split launch from the recorded ncu counters, scaled
    to this launch (reads in proportion to the algorithmic bytes, partial
    writes to the pieces), or None when the kernel's sources differ from the
    ones the counters were taken on."""
    import hashlib

    rec = SPLIT_DRAM
    if not rec.get("sha"):
        return None
    h = hashlib.sha256()
    for f in rec["sources"]:
        with open(os.path.join(ROOT, "paged_fp8_kv_append_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    if h.hexdigest()[:16] != rec["sha"]:
        return None
    return rec["read_per_alg_byte"] * alg_bytes + rec["write_per_piece"] * pieces


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=25.0)
    ap.add_argument("--detail", default="",
                    help="also write every measured line (JSON) to this file")
    ap.add_argument("--no-bf16", action="store_true")
    ap.add_argument("--no-latent", action="store_true")
    ap.add_argument("--no-overhead", action="store_true",
                    help="skip the CUDA-graph verify-overhead measurements")
    ap.add_argument("--overhead-replays", type=int, default=20)
    ap.add_argument("--no-requant", action="store_true",
                    help="skip the re-quantising scale mode lines")
    ap.add_argument("--no-wide", action="store_true",
                    help="skip the 96 q / 8 kv head (12 rows per kv head) step lines")
    ap.add_argument("--no-churn", action="store_true",
                    help="skip the continuous-batching line")
    ap.add_argument("--no-bulk", action="store_true",
                    help="skip the bulk-append (prefill handoff) lines")
    ap.add_argument("--no-extra", action="store_true",
                    help="only the 128k concurrency configs (headline, sweep) and the CPU leg")
    ap.add_argument("--requests", type=int, default=64,
                    help="requests of 131,072 tokens in the headline step (64 = the workload; "
                         "fewer only for small profiling captures)")
    ap.add_argument("--conc-only", type=int, default=0, metavar="B",
                    help="run only the e4m3 step on B requests of 131,072 tokens and print its "
                         "line (small profiling captures)")
    ap.add_argument("--latent-only", type=int, default=0, metavar="B",
                    help="run only the latent verify workload with B requests and print its "
                         "line (small profiling captures)")
    ap.add_argument("--bulk-only", type=int, default=0, metavar="B",
                    help="run only the bulk (prefill handoff) append of B requests of the GQA "
                         "batch workload into an e4m3 pool and print its line (small "
                         "profiling captures)")
    ap.add_argument("--bulk-dtype", type=int, default=0, choices=[0, 1],
                    help="pool dtype of --bulk-only (0 e4m3, 1 bf16)")
    ap.add_argument("--bulk-latent-only", type=int, default=0, metavar="B",
                    help="run only the bulk append of B requests of the latent verify "
                         "workload into an e4m3 pool and print its line (small profiling "
                         "captures)")
    ap.add_argument("--wide-only", type=int, default=0, metavar="B",
                    help="run only the 96 q / 8 kv head step on B requests of the GQA batch "
                         "workload and print its line (small profiling captures)")
    ap.add_argument("--batch", type=int, default=32,
                    help="requests of the GQA batch workload to use (32 = the full workload; "
                         "fewer only for small profiling captures)")
    args = ap.parse_args()
    ws, rank, local = dist_env()
    if args.warmup < 3:
        raise SystemExit("warmup must be >= 3")

    if args.impl == "reference":
        reference_arm(args)
        return

    peaks = _peaks()
    peak = float(peaks.get("hbm_gbs", 6800.0))
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"

    if args.conc_only > 0:
        device = torch.device("cuda", local)
        w = wl.concurrency(args.conc_only)
        w.steps = 3 * (args.steps + args.warmup) + 2
        w.num_pages = int(w.B * (-(-(131072 + w.steps) // 16))) + 64
        arm = Arm(w, 0, device, 3 * (args.steps + args.warmup))
        print(json.dumps(step_line(w, arm, 0, args.steps, args.warmup)))
        return
    if args.wide_only > 0:
        device = torch.device("cuda", local)
        print(json.dumps(wide_group_line(device, args.steps, args.warmup, peak,
                                         B=args.wide_only)))
        return
    if args.bulk_only > 0:
        device = torch.device("cuda", local)
        w = wl.subset(wl.gqa_batch(), args.bulk_only)
        for _ in range(args.warmup):
            bulk_append_line(w, args.bulk_dtype, device, peak)
        print(json.dumps([bulk_append_line(w, args.bulk_dtype, device, peak)
                          for _ in range(args.steps)]))
        return
    if args.bulk_latent_only > 0:
        device = torch.device("cuda", local)
        w = wl.subset(wl.latent_verify(), args.bulk_latent_only)
        for _ in range(args.warmup):
            bulk_append_line(w, 0, device, peak)
        print(json.dumps([bulk_append_line(w, 0, device, peak) for _ in range(args.steps)]))
        return
    if args.latent_only > 0:
        device = torch.device("cuda", local)
        print(json.dumps(latent_bench(args.steps, args.warmup, device, peaks,
                                      B=args.latent_only)))
        return

    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    K, W, R = args.steps, args.warmup, args.overhead_replays
    detail, parity_samples = {}, []
    run_extra = not args.no_extra

    # ---- headline: B requests of 131,072 tokens, e4m3 cache
    B = args.requests
    sweep_pts = [b for b in (1, 8, 16, 32) if b < B]
    head_steps = 1 + 6 * (K + W) + 3 * len(sweep_pts) * (K + W)
    over_steps = 0 if args.no_overhead else 2 * overhead_tokens(R) + 2
    w = wl.concurrency(B, seed=shard_seed(20264, rank))
    w.steps = head_steps + over_steps + 4
    w.num_pages = int(B * (-(-(131072 + w.steps) // 16))) + 64
    arm = Arm(w, 0, device, head_steps)
    rng = np.random.default_rng(w.seed + 5)
    picks = sorted({0, int(rng.integers(1, B))}) if B > 1 else [0]
    pairs = [(r, int(rng.integers(0, w.num_kv_heads))) for r in picks]
    parity_samples.append({"name": "concurrency64_e4m3", "w": w, "dtype": 0, "headline": True,
                           "pairs": pairs, "outs": arm.first_step_output(picks)})
    sampler = ClockSampler(smi_index(local))
    total_ms, per, lens_timed, launches = arm.run(K, W)
    graph_ms = arm.run_graphs(K, W)
    clocks = sampler.stop()
    e2e_ms, h2d, d2h = arm.run_e2e(K, W, graph=True)
    e2e_eager_ms, _, _ = arm.run_e2e(K, W, graph=False)
    # the attention call as one interval (no event between split and combine)
    _, per_attn, lens_attn, _ = arm.run(K, W, split_event=False)
    graph_noattn_ms = arm.run_graphs(K, W, attention=False)
    conc_e4m3 = sweep_lines(w, arm, 0, K, W, peak, sweep_pts)
    overhead = {}
    if not args.no_overhead:
        for b in (1, 8):
            if b <= B:
                overhead[f"concurrency_{b}"] = graph_overhead(arm, R, B=b)
    del arm
    torch.cuda.empty_cache()

    eager_ms = reduce_max(total_ms)
    max_ms = reduce_max(graph_ms)
    tokens = reduce_sum(K * w.B * w.q_tokens)
    value = tokens / (max_ms / 1e3)
    split_ms = per[:, 2]
    attn_ms = per_attn[:, 2]
    attn_bytes = [algorithmic_bytes(w, L, 0) for L in lens_attn]
    split_bytes = [algorithmic_bytes(w, L, 0, include_out=False) for L in lens_timed]
    achieved = float(np.mean([b / (t * 1e6) for b, t in zip(split_bytes, split_ms)]))
    attn_gbs = float(np.mean([b / (t * 1e6) for b, t in zip(attn_bytes, attn_ms)]))
    attn_graph_us = (graph_ms - graph_noattn_ms) / K * 1e3
    head_line = {"requests": B, "attended": B, "tokens_per_s": value,
                 "attn_us_graph": attn_graph_us,
                 "attn_gbs_graph": float(np.mean(attn_bytes)) / (attn_graph_us * 1e3),
                 "ms_per_step": max_ms / K, "eager_ms_per_step": eager_ms / K,
                 "attn_us": float(attn_ms.mean() * 1e3),
                 "attn_gbs": attn_gbs, "pct_of_8000": 100.0 * attn_gbs / NOMINAL_HBM_GBS,
                 "pct_of_measured": 100.0 * attn_gbs / peak,
                 "kernel_us": {k: float(per[:, i].mean() * 1e3)
                               for i, k in enumerate(("append", "verify", "split", "combine"))}}
    conc_e4m3.append(head_line)
    detail["concurrency_e4m3"] = conc_e4m3
    detail["verify_overhead"] = overhead

    # ---- the same requests over a BF16 cache
    conc_bf16 = []
    if not args.no_bf16:
        arm16 = Arm(w, 1, device, 1 + 3 * (len(sweep_pts) + 1) * (K + W))
        parity_samples.append({"name": "concurrency64_bf16", "w": w, "dtype": 1,
                               "pairs": pairs[:1], "outs": arm16.first_step_output(picks[:1])})
        conc_bf16 = sweep_lines(w, arm16, 1, K, W, peak, sweep_pts + [B])
        del arm16
        torch.cuda.empty_cache()
        detail["concurrency_bf16"] = conc_bf16

    gqa = skewed = latent = requant = bulk = wide = churn = handoff = None
    if run_extra:
        # ---- GQA batch (32 requests, 4k..32k), e4m3 and bf16
        gsteps = 1 + 3 * (K + W)
        gw = wl.gqa_batch(seed=shard_seed(20262, rank), steps=gsteps + over_steps + 2)
        if args.batch != gw.B:
            gw = wl.subset(gw, args.batch)
        garm = Arm(gw, 0, device, gsteps)
        rg = int(np.argmax(gw.lens))
        parity_samples.append({"name": "gqa_batch_e4m3", "w": gw, "dtype": 0,
                               "pairs": [(rg, 5)], "outs": garm.first_step_output([rg])})
        g_ms, g_per, g_lens, _ = garm.run(K, W)
        g_graph_ms = garm.run_graphs(K, W)
        g_noattn_ms = garm.run_graphs(K, W, attention=False)
        if not args.no_overhead:
            overhead["gqa_batch"] = graph_overhead(garm, R)
        del garm
        torch.cuda.empty_cache()
        g_attn = g_per[:, 2] + g_per[:, 3]
        g_gbs = float(np.mean([algorithmic_bytes(gw, L, 0) / (t * 1e6)
                               for L, t in zip(g_lens, g_attn)]))
        g_attn_graph_us = (g_graph_ms - g_noattn_ms) / K * 1e3
        g_gbs_graph = float(np.mean([algorithmic_bytes(gw, L, 0) for L in g_lens])) / (
            g_attn_graph_us * 1e3)
        gqa = {"e4m3": {"tokens_per_s": K * gw.B / (g_graph_ms / 1e3),
                        "eager_tokens_per_s": K * gw.B / (g_ms / 1e3),
                        "attn_us": float(g_attn.mean() * 1e3), "attn_gbs": g_gbs,
                        "attn_us_graph": g_attn_graph_us, "attn_gbs_graph": g_gbs_graph,
                        "pct_of_measured": 100.0 * g_gbs / peak,
                        "kernel_us": {k: float(g_per[:, i].mean() * 1e3) for i, k in
                                      enumerate(("append", "verify", "split", "combine"))}}}
        if not args.no_bf16:
            garm16 = Arm(gw, 1, device, 1 + 3 * (K + W))
            parity_samples.append({"name": "gqa_batch_bf16", "w": gw, "dtype": 1,
                                   "pairs": [(rg, 2)], "outs": garm16.first_step_output([rg])})
            gqa["bf16"] = step_line(gw, garm16, 1, K, W)
            gqa["bf16"]["pct_of_measured"] = 100.0 * gqa["bf16"]["attn_gbs"] / peak
            del garm16
            torch.cuda.empty_cache()
        detail["gqa_batch"] = gqa

        # ---- skewed stress workload: verify overhead (the step it is defined
        # on) and the full step with its stale tags
        if not args.no_overhead:
            overhead["skewed"], skewed = skewed_lines(device, R, K, W, peak, parity_samples)
            detail["skewed_step"] = skewed

        if not args.no_latent:
            latent = latent_bench(K, W, device, peaks)
            detail["latent_verify"] = latent
        if not args.no_requant:
            requant = requant_lines(device, K, W, gw)
            detail["requantize"] = requant
        if not args.no_bulk:
            bulk = [bulk_append_line(gw, 0, device, peak), bulk_append_line(gw, 1, device, peak),
                    bulk_append_line(wl.latent_verify(), 0, device, peak)]
            detail["bulk_append"] = bulk
            handoff = [handoff_line(wl.gqa_batch(), device, peak),
                       handoff_line(wl.latent_verify(), device, peak)]
            detail["handoff"] = handoff
        if not args.no_wide:
            wide = {"e4m3": wide_group_line(device, K, W, peak, parity=parity_samples)}
            if not args.no_bf16:
                wide["bf16"] = wide_group_line(device, K, W, peak, dtype=1, parity=parity_samples)
            detail["wide_group"] = wide
        if not args.no_churn:
            churn = churn_line(device, K, W)
            detail["churn"] = churn

    # ---- CPU oracle baseline and parity of the sampled outputs (rank 0)
    cpu, parity = None, {}
    if rank == 0 and args.cpu_budget > 0:
        n_tok, sec, names, parity = cpu_baseline_leg(parity_samples, device, args.cpu_budget)
        cpu = {"value": n_tok / sec, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": f"first decode step of {len(names)} (request, kv head) pair(s) of the "
                         f"headline workload ({', '.join(names)}), each 1/8 of a request's "
                         f"token; {sec:.1f} s on one host core",
               "parity": parity}
        detail["parity"] = parity

    if rank != 0:
        return
    if args.detail:
        with open(args.detail, "w") as fh:
            json.dump(detail, fh)
    # (CTA, segment) pieces: the e4m3 kernel takes 4 of the 8 kv heads per
    # unit, so each request is 2 segments, plus at most one boundary per CTA
    pieces = B * (w.num_kv_heads // 4) + 152
    traffic = split_traffic(float(np.mean(split_bytes)), pieces)
    points = {"concurrency_e4m3": {str(l["requests"]): _pt(l, peak) for l in conc_e4m3}}
    if conc_bf16:
        points["concurrency_bf16"] = {str(l["requests"]): _pt(l, peak) for l in conc_bf16}
    if skewed:
        points["skewed_e4m3"] = _pt(skewed, peak)
    if gqa:
        points["gqa_batch_e4m3"] = _pt(gqa["e4m3"], peak)
        if "bf16" in gqa:
            points["gqa_batch_bf16"] = _pt(gqa["bf16"], peak)
    if wide:
        points["wide96_e4m3"] = _pt(wide["e4m3"], peak)
        if "bf16" in wide:
            points["wide96_bf16"] = _pt(wide["bf16"], peak)
    if latent:
        points["latent_tc"] = {"tok_s": round(latent["value"], 1),
                               "tflops": round(latent["attn_tflops"], 1),
                               "frac": round(latent["tensor_frac"], 4)}
    if overhead:
        points["verify_overhead_pct"] = {k: round(v["verify_overhead_pct"], 2)
                                         for k, v in overhead.items()}
        points["fused_check_overhead_pct"] = {k: round(v["fused_overhead_pct"], 2)
                                              for k, v in overhead.items()}
    if bulk:
        points["bulk_append_frac"] = {f"{b_['workload']}_{b_['cache']}":
                                      round(b_["pct_of_measured"] / 100.0, 4) for b_ in bulk}
    if handoff:
        points["handoff_frac"] = {b_["workload"]: round(b_["pct_of_measured"] / 100.0, 4)
                                  for b_ in handoff}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K,
        "warmup": W, "ms_per_step": max_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 KV, f16 MMA, f32 accumulate",
        "data": "synthetic",
        "config": {"workload": HEADLINE_NAME if B == 64 else f"concurrency {B} x 131072, e4m3",
                   "requests": B, "context": 131072, "q_heads": 64, "kv_heads": 8,
                   "head_dim": 128, "page": 16,
                   "step": "append 1 token/request, tag check, split-K attention, combine; "
                           "each step a CUDA graph replay",
                   "kv_bytes_per_step": int(np.mean(attn_bytes)),
                   "l2": "inputs larger than L2 (KV read per step >> 129 MB)",
                   "parallelism": f"dp{ws} replicas" if ws > 1 else "1 GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "paged_decode_attn_split (plan + gqa_split_kernel<e4m3>)",
                     "achieved_def": "K/V rows + scales + page-table entries + Q over the "
                                     "plan+split CUDA-event time",
                     "algorithmic_bytes": float(np.mean(split_bytes)),
                     "peak_source": peak_src,
                     "attn": {"achieved": attn_gbs, "frac": attn_gbs / peak,
                              "frac_8000": attn_gbs / NOMINAL_HBM_GBS,
                              "def": "K/V + scales + page table + Q + O over split+combine"},
                     "points": points},
        "cpu_baseline": cpu,
        "e2e": {"value": tokens / (reduce_max(e2e_ms) / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "mode": "per step: H2D of its rows and queries, kv_decode_step, D2H of output "
                        "and abort mask; CUDA graph per step",
                "eager_value": tokens / (reduce_max(e2e_eager_ms) / 1e3)},
        "gpu_launches": launches,
        "clocks": clocks,
        "eager_value": tokens / (eager_ms / 1e3),
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
