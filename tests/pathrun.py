"""Test helpers: run one workload through the CUDA library and through the
oracle on identical seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as wl

TOL_ABS, TOL_REL = 2e-3, 1e-2  # attention output tolerance: |o - r| <= abs + rel * |r|


def close(got: np.ndarray, ref: np.ndarray):
    """Elementwise |got - ref| <= 2e-3 + 1e-2 |ref|; returns (ok, max_abs, max_rel, worst)."""
    err = np.abs(got.astype(np.float64) - ref)
    bound = TOL_ABS + TOL_REL * np.abs(ref)
    ok = bool(np.all(err <= bound))
    rel = err / np.maximum(np.abs(ref), 1e-30)
    worst = float(np.max(err - bound)) if err.size else 0.0
    return ok, float(err.max(initial=0.0)), float(rel.max(initial=0.0)), worst


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
        torch.bfloat16).to(torch.float64).numpy()


class Both:
    """A pool on the device (library) and its host twin (oracle)."""

    def __init__(self, w: wl.Workload, dtype: int, device="cuda", num_pages=None, free=None,
                 tags=None, scale_mode=0):
        import paged_fp8_kv_append_gb300 as kv

        self.kv, self.w, self.dtype = kv, w, dtype
        npg = num_pages or w.num_pages
        free = wl.free_list(w) if free is None else free
        tags = wl.initial_tags(w) if tags is None else tags
        self.dev = kv.KVPool(npg, w.page_size, w.num_kv_heads, w.head_dim_k, w.head_dim_v,
                             dtype=dtype, layout=w.layout, device=device, tags=tags,
                             free_list=free, scale_mode=scale_mode)
        self.ref = oracle.Pool(npg, w.page_size, w.num_kv_heads, w.head_dim_k, w.head_dim_v,
                               dtype=dtype, layout=w.layout, tags=tags, free_list=free,
                               scale_mode=scale_mode)
        B, mp = w.B, w.max_pages
        self.pt_d = torch.full((B, mp), -1, dtype=torch.int32, device=device)
        self.et_d = torch.zeros((B, mp), dtype=torch.int32, device=device)
        self.sl_d = torch.zeros(B, dtype=torch.int32, device=device)
        self.pt_h = np.full((B, mp), -1, np.int32)
        self.et_h = np.zeros((B, mp), np.uint32)
        self.sl_h = np.zeros(B, np.int32)
        self.device = device

    def append(self, rows_k, rows_v, counts, max_new=None):
        """Append per-request rows (lists of bf16 device tensors) on both sides."""
        B = self.w.B
        counts = np.asarray(counts, np.int64)
        ind = np.zeros(B + 1, np.int32)
        ind[1:] = np.cumsum(counts)
        k = torch.cat([x for x in rows_k if x is not None and x.shape[0] > 0]) if ind[-1] else None
        v = None
        if self.w.layout == 0 and ind[-1]:
            v = torch.cat([x for x in rows_v if x is not None and x.shape[0] > 0])
        mx = int(counts.max()) if max_new is None else max_new
        ind_d = torch.from_numpy(ind).to(self.device)
        if k is None:  # nothing to append: still a valid call
            k = torch.zeros((1, self.w.num_kv_heads, self.w.head_dim_k), dtype=torch.bfloat16,
                            device=self.device)
            v = torch.zeros((1, self.w.num_kv_heads, self.w.head_dim_v), dtype=torch.bfloat16,
                            device=self.device) if self.w.layout == 0 else None
        self.dev.append(B, k.contiguous(), None if v is None else v.contiguous(), ind_d, mx,
                        self.pt_d, self.et_d, self.sl_d)
        kb = wl.bits_u16(k)
        vb = wl.bits_u16(v) if v is not None else None
        st, stop = oracle.append(self.ref, kb, vb, ind, mx, self.pt_h, self.et_h, self.sl_h)
        return st, stop

    def fill(self, lens=None, tag=0):
        w = self.w
        lens = w.lens if lens is None else lens
        ks, vs = [], []
        for r in range(w.B):
            k, v = wl.kv_rows(w, r, int(self.sl_h[r]), int(lens[r]), device=self.device, tag=tag)
            ks.append(k)
            vs.append(v)
        return self.append(ks, vs, lens)

    def make_stale(self):
        """Give the workload's stale requests one stale expected tag (both sides)."""
        for r, j in wl.stale_slots(self.w):
            self.et_h[r, j] = np.uint32(self.et_h[r, j]) - np.uint32(1)
        self.et_d.copy_(torch.from_numpy(self.et_h.view(np.int32)))

    def release(self, mask=None):
        """Release the masked requests' pages (all when mask is None) on both
        sides; returns the oracle's status (the device's goes to ctl)."""
        B = self.w.B
        ws = torch.empty(self.kv.kv_release_workspace_size(B), dtype=torch.uint8,
                         device=self.device)
        m = None if mask is None else np.asarray(mask, np.uint8)
        m_d = None if m is None else torch.from_numpy(m).to(self.device)
        self.dev.release(B, self.pt_d, self.et_d, self.sl_d, m_d, ws)
        return oracle.release(self.ref, self.pt_h, self.et_h, self.sl_h, m)

    # ---- state comparison (bit-exact)
    def assert_state_equal(self):
        d, r = self.dev, self.ref
        kc = d.k_cache.cpu()
        if self.dtype == 1:
            kc = kc.view(torch.int16)
        assert np.array_equal(kc.numpy().view(r.k_cache.dtype), r.k_cache), "k_cache"
        if r.v_cache is not None:
            vc = d.v_cache.cpu()
            if self.dtype == 1:
                vc = vc.view(torch.int16)
            assert np.array_equal(vc.numpy().view(r.v_cache.dtype), r.v_cache), "v_cache"
        if self.dtype == 0:
            assert np.array_equal(d.k_scale.cpu().numpy().view(np.uint32),
                                  r.k_scale.view(np.uint32)), "k_scale"
            if r.v_scale is not None:
                assert np.array_equal(d.v_scale.cpu().numpy().view(np.uint32),
                                      r.v_scale.view(np.uint32)), "v_scale"
        assert np.array_equal(d.tags.cpu().numpy().view(np.uint32), r.tags), "tags"
        assert np.array_equal(self.pt_d.cpu().numpy(), self.pt_h), "page_table"
        assert np.array_equal(self.et_d.cpu().numpy().view(np.uint32), self.et_h), "exp_tags"
        assert np.array_equal(self.sl_d.cpu().numpy(), self.sl_h), "seq_lens"
        assert int(d.ctl[0].item()) == int(r.free_head[0]), "free_head"
        assert np.array_equal(d.free_list.cpu().numpy(), r.free_list), "free_list"

    def verify(self):
        B = self.w.B
        m_d = torch.zeros(B, dtype=torch.uint8, device=self.device)
        self.dev.verify(B, self.pt_d, self.et_d, self.sl_d, m_d)
        m_h = oracle.verify(self.ref.num_pages, self.w.page_size, self.ref.tags, self.pt_h,
                            self.et_h, self.sl_h)
        return m_d, m_h

    def step(self, leave, rows_k, rows_v, counts, q, remove=True, max_new=None, sentinel=7.0):
        """One kv_decode_step on the device and oracle.step on the host, on
        the same rows (lists of per-request bf16 device tensors) and queries.
        Returns (oracle status, device abort mask, oracle abort mask, device
        out, oracle out, oracle written)."""
        w, B = self.w, self.w.B
        counts = np.asarray(counts, np.int64)
        ind = np.zeros(B + 1, np.int32)
        ind[1:] = np.cumsum(counts)
        ks = [x for x in rows_k if x is not None and x.shape[0] > 0]
        vs = [x for x in rows_v if x is not None and x.shape[0] > 0] if w.layout == 0 else []
        if ks:
            k = torch.cat(ks).contiguous()
            v = torch.cat(vs).contiguous() if w.layout == 0 else None
        else:  # nothing to append: still a valid call
            k = torch.zeros((1, w.num_kv_heads, w.head_dim_k), dtype=torch.bfloat16,
                            device=self.device)
            v = torch.zeros((1, w.num_kv_heads, w.head_dim_v), dtype=torch.bfloat16,
                            device=self.device) if w.layout == 0 else None
        mx = int(counts.max()) if max_new is None else max_new
        lv = None if leave is None else np.asarray(leave, np.uint8)
        lv_d = None if lv is None else torch.from_numpy(lv).to(self.device)
        out = torch.full((B, w.q_tokens, w.num_q_heads, w.head_dim_v), sentinel,
                         dtype=torch.bfloat16, device=self.device)
        m_d = torch.full((B,), 0xEE, dtype=torch.uint8, device=self.device)
        ws = torch.empty(self.dev.step_workspace_size(B, w.num_q_heads, w.q_tokens),
                         dtype=torch.uint8, device=self.device)
        flags = self.kv.KV_STEP_REMOVE_ABORTED if remove else 0
        self.dev.step(B, w.num_q_heads, w.q_tokens, lv_d, k, v, torch.from_numpy(ind).to(self.device),
                      mx, self.pt_d, self.et_d, self.sl_d, q, w.sm_scale, out, m_d, flags, ws)
        st, m_h, ref, written = oracle.step(
            self.ref, lv, wl.bits_u16(k), None if v is None else wl.bits_u16(v), ind, mx,
            self.pt_h, self.et_h, self.sl_h, wl.bits_u16(q), w.sm_scale, w.num_q_heads,
            w.q_tokens, remove_aborted=remove)
        return st, m_d, m_h, out, ref, written

    def attn(self, q, abort_d, abort_h, sentinel=7.0, phases=False):
        w, B = self.w, self.w.B
        out = torch.full((B, w.q_tokens, w.num_q_heads, w.head_dim_v), sentinel,
                         dtype=torch.bfloat16, device=self.device)
        ws = torch.empty(self.dev.workspace_size(B, w.num_q_heads, w.q_tokens), dtype=torch.uint8,
                         device=self.device)
        if phases:
            self.kv.paged_decode_attn_split(self.dev.handle, B, w.num_q_heads, w.q_tokens, q,
                                            self.pt_d, self.sl_d, abort_d, w.sm_scale, ws)
            self.kv.paged_decode_attn_combine(self.dev.handle, B, w.num_q_heads, w.q_tokens,
                                              abort_d, out, ws)
        else:
            self.dev.attn(B, w.num_q_heads, w.q_tokens, q, self.pt_d, self.sl_d, abort_d,
                          w.sm_scale, out, ws)
        ref, written = oracle.attn(self.ref, wl.bits_u16(q), self.pt_h, self.sl_h, abort_h,
                                   w.sm_scale, w.num_q_heads, w.q_tokens)
        return out, ref, written


class Bookkeeping:
    """Host twin of a pool's integer state (tags, free list, free head) for
    oracle.alloc / oracle.verify, without the cache arrays."""

    def __init__(self, num_pages, page_size, tags, free_list):
        self.num_pages, self.page_size = int(num_pages), int(page_size)
        self.tags = np.array(tags, dtype=np.uint32)
        self.free_list = np.array(free_list, dtype=np.int32)
        self.free_head = np.zeros(1, np.int32)


class FullSize:
    """A full-size workload on the device, with the oracle twinning every
    request's bookkeeping and, for sampled (request, kv head) pairs, the cache
    contents and attention output (a one-kv-head oracle pool fed the same rows
    in the same calls)."""

    def __init__(self, w: wl.Workload, dtype: int, device="cuda", sample=(), heads=(0,)):
        import paged_fp8_kv_append_gb300 as kv

        self.kv, self.w, self.dtype, self.device = kv, w, dtype, device
        tags, free = wl.initial_tags(w), wl.free_list(w)
        self.dev = kv.KVPool(w.num_pages, w.page_size, w.num_kv_heads, w.head_dim_k,
                             w.head_dim_v, dtype=dtype, layout=w.layout, device=device, tags=tags,
                             free_list=free)
        self.bk = Bookkeeping(w.num_pages, w.page_size, tags, free)
        B, mp = w.B, w.max_pages
        self.pt_d = torch.full((B, mp), -1, dtype=torch.int32, device=device)
        self.et_d = torch.zeros((B, mp), dtype=torch.int32, device=device)
        self.sl_d = torch.zeros(B, dtype=torch.int32, device=device)
        self.pt_h = np.full((B, mp), -1, np.int32)
        self.et_h = np.zeros((B, mp), np.uint32)
        self.sl_h = np.zeros(B, np.int32)
        # oracle twins: (r, h) -> (pool, page table, exp tags, seq len)
        self.sample, self.heads = list(sample), list(heads)
        self.twins = {}
        for r in self.sample:
            for h in self.heads:
                npg = int(-(-(int(w.lens[r]) + w.steps) // w.page_size)) + 2
                pool = oracle.Pool(npg, w.page_size, 1, w.head_dim_k, w.head_dim_v, dtype=dtype)
                self.twins[(r, h)] = [pool, np.full((1, npg), -1, np.int32),
                                      np.zeros((1, npg), np.uint32), np.zeros(1, np.int32)]

    def _append(self, ks, vs, counts, max_new):
        """One append call: ks/vs lists (per request, device bf16 [n][Hkv][D])."""
        B = self.w.B
        counts = np.asarray(counts, np.int64)
        ind = np.zeros(B + 1, np.int32)
        ind[1:] = np.cumsum(counts)
        k = torch.cat([x for x in ks if x is not None and x.shape[0] > 0])
        v = torch.cat([x for x in vs if x is not None and x.shape[0] > 0])
        self.dev.append(B, k, v, torch.from_numpy(ind).to(self.device), int(max_new), self.pt_d,
                        self.et_d, self.sl_d)
        st, stop = oracle.alloc(self.bk, ind, int(max_new), self.pt_h, self.et_h, self.sl_h)
        for (r, h), tw in self.twins.items():
            if counts[r] == 0:
                continue
            pool, pt, et, sl = tw
            kb = wl.bits_u16(ks[r][:, h:h + 1, :])
            vb = wl.bits_u16(vs[r][:, h:h + 1, :])
            s2, _ = oracle.append(pool, kb, vb, np.array([0, counts[r]], np.int32), int(counts[r]),
                                  pt, et, sl)
            assert s2 == 0
        return st, stop

    def fill(self, group=4):
        """Every request's first L_r - 1 tokens, `group` requests per call."""
        w = self.w
        for r0 in range(0, w.B, group):
            counts = np.zeros(w.B, np.int64)
            ks, vs = [None] * w.B, [None] * w.B
            for r in range(r0, min(w.B, r0 + group)):
                counts[r] = int(w.lens[r]) - 1
                ks[r], vs[r] = wl.kv_rows(w, r, 0, int(counts[r]), device=self.device)
            st, stop = self._append(ks, vs, counts, int(counts.max()))
            assert (st, stop) == (0, w.B)

    def step_append(self, s):
        k, v = wl.step_rows(self.w, s, device=self.device)
        ks = [k[r:r + 1] for r in range(self.w.B)]
        vs = [v[r:r + 1] for r in range(self.w.B)]
        return self._append(ks, vs, np.ones(self.w.B, np.int64), 1)

    def make_stale(self):
        for r, j in wl.stale_slots(self.w):
            self.et_h[r, j] = np.uint32(self.et_h[r, j]) - np.uint32(1)
        self.et_d.copy_(torch.from_numpy(self.et_h.view(np.int32)))

    def assert_bookkeeping(self):
        d = self.dev
        assert np.array_equal(d.tags.cpu().numpy().view(np.uint32), self.bk.tags), "tags"
        assert np.array_equal(self.pt_d.cpu().numpy(), self.pt_h), "page_table"
        assert np.array_equal(self.et_d.cpu().numpy().view(np.uint32), self.et_h), "exp_tags"
        assert np.array_equal(self.sl_d.cpu().numpy(), self.sl_h), "seq_lens"
        assert int(d.ctl[0].item()) == int(self.bk.free_head[0]), "free_head"

    def assert_sampled_cache(self):
        """Cache bytes and scales of every sampled (request, kv head), by logical page."""
        P = self.w.page_size
        for (r, h), (pool, pt, et, sl) in self.twins.items():
            n = int(-(-int(sl[0]) // P))
            assert int(sl[0]) == int(self.sl_h[r])
            pages_d = torch.from_numpy(self.pt_h[r, :n].astype(np.int64)).to(self.device)
            kc = self.dev.k_cache[pages_d, h].cpu()
            vc = self.dev.v_cache[pages_d, h].cpu()
            if self.dtype == 1:
                kc, vc = kc.view(torch.int16), vc.view(torch.int16)
            want_k = pool.k_cache[pt[0, :n], 0]
            want_v = pool.v_cache[pt[0, :n], 0]
            assert np.array_equal(kc.numpy().view(want_k.dtype), want_k), (r, h, "k")
            assert np.array_equal(vc.numpy().view(want_v.dtype), want_v), (r, h, "v")
            if self.dtype == 0:
                ks = self.dev.k_scale[pages_d, h].cpu().numpy()
                vs = self.dev.v_scale[pages_d, h].cpu().numpy()
                assert np.array_equal(ks.view(np.uint32), pool.k_scale[pt[0, :n], 0].view(np.uint32))
                assert np.array_equal(vs.view(np.uint32), pool.v_scale[pt[0, :n], 0].view(np.uint32))

    def verify(self):
        B = self.w.B
        m_d = torch.zeros(B, dtype=torch.uint8, device=self.device)
        self.dev.verify(B, self.pt_d, self.et_d, self.sl_d, m_d)
        m_h = oracle.verify(self.bk.num_pages, self.w.page_size, self.bk.tags, self.pt_h,
                            self.et_h, self.sl_h)
        return m_d, m_h

    def attn_check(self, q, abort_d, abort_h, sentinel=7.0, fused=False):
        """Attention on the device for the whole batch; oracle for the samples.
        fused: the call with the tag check inside its page reads
        (paged_decode_attn_checked), whose abort mask must equal abort_h."""
        w, B = self.w, self.w.B
        out = torch.full((B, w.q_tokens, w.num_q_heads, w.head_dim_v), sentinel,
                         dtype=torch.bfloat16, device=self.device)
        ws = torch.empty(self.dev.workspace_size(B, w.num_q_heads, w.q_tokens), dtype=torch.uint8,
                         device=self.device)
        if fused:
            mask = torch.full((B,), 0xEE, dtype=torch.uint8, device=self.device)
            self.kv.paged_decode_attn_checked(self.dev.handle, B, w.num_q_heads, w.q_tokens, q,
                                              self.pt_d, self.et_d, self.sl_d, w.sm_scale, out,
                                              mask, ws)
            want = np.zeros(B, np.uint8) if abort_h is None else np.asarray(abort_h, np.uint8)
            assert np.array_equal(mask.cpu().numpy(), want), "fused check's abort mask"
        else:
            self.dev.attn(B, w.num_q_heads, w.q_tokens, q, self.pt_d, self.sl_d, abort_d,
                          w.sm_scale, out, ws)
        got = bf16_to_f64(out.cpu().view(torch.int16).numpy().view(np.uint16))
        G = w.num_q_heads // w.num_kv_heads
        qh = q.cpu()
        checked = 0
        jobs, keys = [], []
        for (r, h), (pool, pt, et, sl) in self.twins.items():
            if abort_h is not None and abort_h[r]:
                assert np.all(got[r] == sentinel), f"aborted request {r} written"
                continue
            qs = wl.bits_u16(qh[r:r + 1, :, h * G:(h + 1) * G, :])
            jobs.append((pool, qs, pt, sl, w.sm_scale, G, w.q_tokens))
            keys.append((r, h))
        if len(jobs) > 8:  # many long twins: the oracle in a spawn-started process pool
            import multiprocessing as mp
            import os

            with mp.get_context("spawn").Pool(min(16, os.cpu_count() or 1)) as workers:
                refs = workers.map(gqa_oracle_attn, jobs)
        else:
            refs = [gqa_oracle_attn(j) for j in jobs]
        for (r, h), ref in zip(keys, refs):
            ok, mabs, mrel, _ = close(got[r, :, h * G:(h + 1) * G], ref)
            assert ok, (r, h, mabs, mrel)
            checked += 1
        if abort_h is not None:
            for r in np.nonzero(abort_h)[0]:
                assert np.all(got[r] == sentinel), f"aborted request {r} written"
        return checked


def latent_oracle_request(args):
    """One latent request in the oracle, for a process pool (started with
    spawn): its rows appended to a fresh one-request pool, then every head
    and draft token attended.  Returns (cache codes by logical page, scales,
    attention output [T][Hq][Dv])."""
    rows, L, q_bits, sm_scale, Hq, T = args
    npg = -(-L // 64) + 1
    pool = oracle.Pool(npg, 64, 1, 576, 512, dtype=0, layout=1)
    ptr = np.full((1, npg), -1, np.int32)
    slr = np.zeros(1, np.int32)
    st, _ = oracle.append(pool, rows, None, np.array([0, L], np.int32), L, ptr,
                          np.zeros((1, npg), np.uint32), slr)
    assert st == 0
    n = -(-L // 64)
    ref, written = oracle.attn(pool, q_bits, ptr, slr, None, sm_scale, Hq, T)
    assert written[0] == 1
    return pool.k_cache[ptr[0, :n]], pool.k_scale[ptr[0, :n]], ref[0]


def gqa_oracle_attn(args):
    """Oracle attention of one one-kv-head twin pool (picklable, for a process
    pool): returns the output [T][G][Dv] of its request."""
    pool, qs, pt, sl, sm_scale, G, T = args
    ref, written = oracle.attn(pool, qs, pt, sl, None, sm_scale, G, T)
    assert written[0] == 1
    return ref[0]
