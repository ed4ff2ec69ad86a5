"""Seeded synthetic workloads for the paged FP8 KV decode path.

Shared by the tests (which feed the same inputs to the CUDA library and to
the CPU oracle) and by bench.py.  This module holds no arithmetic of the
method: it only draws lengths, page permutations, tags and bf16 K/V/Q values.

The five workloads follow the shapes, sizes and distributions of the decode
benchmark configurations (GQA batch, latent speculative verify, concurrency
sweep, skewed long-context stress).  Where a distribution is given only by its
median (lognormal lengths) the log-space sigma is 1.0.  Host metadata comes
from numpy's PCG64 generator seeded with 20260 + k; bulk values come from a
torch generator on the target device with the same seed, drawn in fp32 and
rounded to bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass
class Workload:
    name: str
    seed: int
    lens: np.ndarray             # int32 [B]: tokens cached when the step's query runs
    num_q_heads: int
    num_kv_heads: int
    head_dim_k: int
    head_dim_v: int
    page_size: int
    q_tokens: int
    layout: int                  # 0 GQA, 1 latent
    num_pages: int
    sm_scale: float              # fp32 value passed to the kernels
    stale: list = field(default_factory=list)  # requests given one stale expected tag
    channel_std: bool = False    # per-(K|V, head, dim) std ~ U(0.5, 4)
    steps: int = 0               # decode steps the pool must have room for
    magnitude: float = 1.0       # K/V rows are drawn at this overall scale

    @property
    def B(self) -> int:
        return int(len(self.lens))

    @property
    def pages_per_req(self) -> np.ndarray:
        return -(-self.lens.astype(np.int64) // self.page_size)

    @property
    def max_pages(self) -> int:
        return int(-(-(int(self.lens.max()) + self.steps) // self.page_size)) + 1


def _f32(x: float) -> float:
    return float(np.float32(x))


def tiny(seed: int = 20261) -> Workload:
    """4 requests {37, 64, 100, 255}; 8 q heads / 2 kv heads, D 128, P 16, 256
    pages; one stale expected tag in request 2."""
    return Workload("tiny", seed, np.array([37, 64, 100, 255], np.int32), 8, 2, 128, 128, 16,
                    1, 0, 256, _f32(1 / math.sqrt(128)), stale=[2])


def gqa_batch(seed: int = 20262, steps: int = 0) -> Workload:
    """32 requests with contexts uniform in 4k..32k; 64 q / 8 kv heads, D 128,
    P 16; K/V per-channel std ~ U(0.5, 4); pool = pages needed x 1.1."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(4096, 32768, size=32, endpoint=True).astype(np.int32)
    need = int((-(-(lens.astype(np.int64) + steps) // 16)).sum())
    return Workload("gqa_batch", seed, lens, 64, 8, 128, 128, 16, 1, 0, int(math.ceil(need * 1.1)),
                    _f32(1 / math.sqrt(128)), channel_std=True, steps=steps)


def latent_verify(seed: int = 20263, B: int = 64) -> Workload:
    """Latent (MLA-style) speculative verify: lognormal contexts (median 16k)
    clipped to 8k..64k; 128 q heads on one 576-wide kv row (V = first 512),
    P 64, 4 causal query tokens."""
    rng = np.random.default_rng(seed)
    lens = np.clip(np.round(rng.lognormal(math.log(16384), 1.0, size=B)), 8192, 65536)
    lens = lens.astype(np.int32)
    need = int((-(-lens.astype(np.int64) // 64)).sum())
    return Workload("latent_verify", seed, lens, 128, 1, 576, 512, 64, 4, 1,
                    int(math.ceil(need * 1.1)) + 8, _f32(1 / math.sqrt(576)))


def concurrency(B: int, seed: int = 20264) -> Workload:
    """B requests of 128k tokens; 64 q / 8 kv heads, D 128, P 16."""
    lens = np.full(B, 131072, np.int32)
    return Workload(f"concurrency_{B}", seed, lens, 64, 8, 128, 128, 16, 1, 0, B * 8192 + 64,
                    _f32(1 / math.sqrt(128)))


def skewed(seed: int = 20265, steps: int = 10) -> Workload:
    """256 requests, lognormal contexts (median 16k) clipped to 1..256k; 32 q /
    4 kv heads, D 128, P 16; pool = pages for all steps x 1.1; 1% stale."""
    rng = np.random.default_rng(seed)
    B = 256
    lens = np.clip(np.round(rng.lognormal(math.log(16384), 1.0, size=B)), 1, 262144)
    lens = lens.astype(np.int32)
    stale = sorted(rng.choice(B, size=int(round(0.01 * B)), replace=False).tolist())
    need = int((-(-(lens.astype(np.int64) + steps) // 16)).sum())
    return Workload("skewed", seed, lens, 32, 4, 128, 128, 16, 1, 0, int(math.ceil(need * 1.1)),
                    _f32(1 / math.sqrt(128)), stale=stale, steps=steps)


# ------------------------------------------------------------------ draws

def free_list(w: Workload) -> np.ndarray:
    """Seeded shuffle of all page ids (the pool's free list)."""
    return np.random.default_rng(w.seed + 1).permutation(w.num_pages).astype(np.int32)


def initial_tags(w: Workload) -> np.ndarray:
    return np.random.default_rng(w.seed + 2).integers(0, 2 ** 32, w.num_pages,
                                                      dtype=np.uint64).astype(np.uint32)


def stale_slots(w: Workload) -> list:
    """(request, logical page) whose expected tag is made stale: one seeded
    page per stale request."""
    rng = np.random.default_rng(w.seed + 3)
    return [(r, int(rng.integers(0, int(w.pages_per_req[r])))) for r in w.stale]


def channel_std(w: Workload, which: int) -> np.ndarray | None:
    """Per-(kv head, dim) std ~ U(0.5, 4) for K (which=0) or V (which=1)."""
    if not w.channel_std:
        return None
    rng = np.random.default_rng(w.seed + 10 + which)
    return rng.uniform(0.5, 4.0, size=(w.num_kv_heads, w.head_dim_k if which == 0 else w.head_dim_v))


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def kv_rows(w: Workload, r: int, row0: int, nrows: int, device="cpu", tag: int = 0):
    """bf16 K and V rows [nrows][Hkv][D] of request r, positions row0.. .

    Each (request, 4096-position block) has its own generator stream, so any
    slice of a request's rows can be regenerated independently and on any
    device of the same kind.  Latent layout: one tensor [nrows][Dk]; V is None.
    """
    if nrows <= 0:
        if w.layout == 1:
            return torch.zeros((0, w.head_dim_k), dtype=torch.bfloat16, device=device), None
        return (torch.zeros((0, w.num_kv_heads, w.head_dim_k), dtype=torch.bfloat16, device=device),
                torch.zeros((0, w.num_kv_heads, w.head_dim_v), dtype=torch.bfloat16, device=device))
    outs_k, outs_v = [], []
    pos = row0
    end = row0 + nrows
    while pos < end:
        blk = pos // 4096
        lo, hi = pos - blk * 4096, min(end - blk * 4096, 4096)
        base = (w.seed * 1_000_003 + r * 7919 + blk * 104729 + tag * 15485863)
        if w.layout == 1:
            x = torch.randn((4096, w.head_dim_k), generator=_gen(base, device), device=device)
            outs_k.append(x[lo:hi])
        else:
            k = torch.randn((4096, w.num_kv_heads, w.head_dim_k), generator=_gen(base, device),
                            device=device)
            v = torch.randn((4096, w.num_kv_heads, w.head_dim_v), generator=_gen(base + 1, device),
                            device=device)
            outs_k.append(k[lo:hi])
            outs_v.append(v[lo:hi])
        pos = blk * 4096 + hi
    k = torch.cat(outs_k)
    if w.layout == 1:
        return (k * w.magnitude).to(torch.bfloat16), None
    v = torch.cat(outs_v)
    sk, sv = channel_std(w, 0), channel_std(w, 1)
    if sk is not None:
        k = k * torch.as_tensor(sk, dtype=torch.float32, device=device)
        v = v * torch.as_tensor(sv, dtype=torch.float32, device=device)
    return (k * w.magnitude).to(torch.bfloat16), (v * w.magnitude).to(torch.bfloat16)


def queries(w: Workload, device="cpu", step: int = 0) -> torch.Tensor:
    """bf16 q [B][T][Hq][Dk] for one decode step."""
    g = _gen(w.seed * 31 + 977 + step, device)
    q = torch.randn((w.B, w.q_tokens, w.num_q_heads, w.head_dim_k), generator=g, device=device)
    return q.to(torch.bfloat16)


def bits_u16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def step_rows(w: Workload, step: int, device="cpu"):
    """bf16 K/V of the one new token every request appends at decode step
    `step`: [B][Hkv][Dk] and [B][Hkv][Dv] (latent: [B][Dk], None)."""
    g = _gen(w.seed * 131 + 7 + step, device)
    if w.layout == 1:
        return torch.randn((w.B, w.head_dim_k), generator=g, device=device).to(torch.bfloat16), None
    k = torch.randn((w.B, w.num_kv_heads, w.head_dim_k), generator=g, device=device)
    v = torch.randn((w.B, w.num_kv_heads, w.head_dim_v), generator=g, device=device)
    sk, sv = channel_std(w, 0), channel_std(w, 1)
    if sk is not None:
        k = k * torch.as_tensor(sk, dtype=torch.float32, device=device)
        v = v * torch.as_tensor(sv, dtype=torch.float32, device=device)
    return k.to(torch.bfloat16), v.to(torch.bfloat16)


def subset(w: Workload, n: int) -> Workload:
    """The first n requests of a workload, with a pool sized to match."""
    import dataclasses

    lens = w.lens[:n].copy()
    need = int((-(-(lens.astype(np.int64) + w.steps) // w.page_size)).sum())
    return dataclasses.replace(w, name=f"{w.name}[:{n}]", lens=lens,
                               num_pages=int(math.ceil(need * 1.1)) + 8,
                               stale=[r for r in w.stale if r < n])
