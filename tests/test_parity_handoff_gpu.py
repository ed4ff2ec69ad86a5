"""GPU parity of kv_append_from_pool, the prefill-to-decode handoff ("Smaller,
faster, safer: running Kimi and GLM at scale", section "Quantizing the KV
cache": prefill keeps a BF16 cache, decode reads an FP8 one).  Rows are
read from a bf16 pool through its page table and appended to another pool;
the destination must equal, bit for bit, the oracle's kv_append_quantize of
the same rows (page pops, tags, page tables, scales, codes), and attention
over it must match the oracle."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from pathrun import Both, bf16_to_f64, close

pytestmark = pytest.mark.gpu


def _workload(layout, seed):
    if layout == 0:
        lens = np.array([37, 64, 100, 255, 0, 16, 1, 4097], np.int32)
        return wl.Workload("handoff", seed, lens, 8, 2, 128, 128, 16, 1, 0, 512,
                           float(np.float32(1 / np.sqrt(128))))
    lens = np.array([37, 300, 64, 1000, 0, 129], np.int32)
    return wl.Workload("handoff_lat", seed, lens, 16, 1, 576, 512, 64, 4, 1, 64,
                       float(np.float32(1 / np.sqrt(576))))


def _rows(w, lens):
    ks, vs = [], []
    for r in range(w.B):
        k, v = wl.kv_rows(w, r, 0, int(lens[r]), device="cuda")
        ks.append(k)
        vs.append(v)
    return ks, vs


def _source(w, ks, vs, check=True):
    """A bf16 pool (its own free list and tags) holding every request's rows
    (checked page by page against the rows when `check`)."""
    import paged_fp8_kv_append_gb300 as kv

    B, mp = w.B, w.max_pages
    rng = np.random.default_rng(w.seed + 99)
    pool = kv.KVPool(w.num_pages, w.page_size, w.num_kv_heads, w.head_dim_k, w.head_dim_v,
                     dtype=kv.KV_DTYPE_BF16, layout=w.layout, device="cuda",
                     tags=rng.integers(0, 2 ** 32, w.num_pages, dtype=np.uint64).astype(np.uint32),
                     free_list=rng.permutation(w.num_pages).astype(np.int32))
    pt = torch.full((B, mp), -1, dtype=torch.int32, device="cuda")
    et = torch.zeros((B, mp), dtype=torch.int32, device="cuda")
    sl = torch.zeros(B, dtype=torch.int32, device="cuda")
    ind = torch.from_numpy(np.concatenate([[0], np.cumsum(w.lens)]).astype(np.int32)).cuda()
    k = torch.cat([x for x in ks if x.shape[0] > 0])
    v = torch.cat([x for x in vs if x.shape[0] > 0]) if w.layout == 0 else None
    pool.append(B, k, v, ind, int(w.lens.max()), pt, et, sl)
    torch.cuda.synchronize()
    assert pool.error() == 0
    # the source holds the rows' bits, page by page through its table
    P, pth = w.page_size, pt.cpu().numpy()
    for r in range(B if check else 0):
        L = int(w.lens[r])
        for j in range(-(-L // P)):
            n = min(P, L - j * P)
            got = pool.k_cache[int(pth[r, j]), :, :n] if w.layout == 0 else \
                pool.k_cache[int(pth[r, j]), :n]
            want = ks[r][j * P:j * P + n].transpose(0, 1) if w.layout == 0 else \
                ks[r][j * P:j * P + n]
            assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    return pool, pt, sl


def _oracle_append(b, ks, vs, lens):
    w = b.w
    ind = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    kb = np.concatenate([wl.bits_u16(x) for x in ks])
    vb = np.concatenate([wl.bits_u16(x) for x in vs]) if w.layout == 0 else None
    return oracle.append(b.ref, kb, vb if vb is not None else kb, ind, int(max(lens.max(), 1)),
                         b.pt_h, b.et_h, b.sl_h)


@pytest.mark.parametrize("layout,dst_dtype", [(0, 0), (0, 1), (1, 0)])
def test_handoff_matches_append_of_the_same_rows(layout, dst_dtype):
    """Ragged lengths (partial last pages, an empty request, exact pages)."""
    w = _workload(layout, 4801 + 10 * layout + dst_dtype)
    ks, vs = _rows(w, w.lens)
    src, spt, ssl = _source(w, ks, vs)
    b = Both(w, dst_dtype)
    b.dev.append_from_pool(w.B, src, spt, ssl, b.pt_d, b.et_d, b.sl_d)
    st, stop = _oracle_append(b, ks, vs, w.lens)
    assert (st, stop) == (0, w.B)
    torch.cuda.synchronize()
    assert b.dev.error() == 0
    b.assert_state_equal()
    if dst_dtype == 0:
        q = wl.queries(w, device="cuda")
        out, ref, written = b.attn(q, None, None)
        got = bf16_to_f64(out.cpu().view(torch.int16).numpy().view(np.uint16))
        for r in range(w.B):
            ok, mabs, mrel, _ = close(got[r], ref[r])
            assert ok, (r, mabs, mrel)


def test_handoff_into_nonempty_request_stops():
    """A request that already holds rows in the destination stops the call
    there (KV_ERR_INVALID_ARG): earlier requests are served, later ones are
    left untouched."""
    import paged_fp8_kv_append_gb300 as kv

    w = _workload(0, 4851)
    ks, vs = _rows(w, w.lens)
    src, spt, ssl = _source(w, ks, vs)
    b = Both(w, 0)
    one = np.zeros(w.B, np.int64)
    one[2] = 5  # request 2 gets 5 rows first
    k2, v2 = wl.kv_rows(w, 2, 0, 5, device="cuda", tag=3)
    rk = [k2 if r == 2 else ks[r][:0] for r in range(w.B)]
    rv = [v2 if r == 2 else vs[r][:0] for r in range(w.B)]
    assert b.append(rk, rv, one)[0] == 0
    b.dev.append_from_pool(w.B, src, spt, ssl, b.pt_d, b.et_d, b.sl_d)
    served = w.lens.copy()
    served[2:] = 0
    st, stop = _oracle_append(b, ks, vs, served)
    assert st == 0
    torch.cuda.synchronize()
    assert b.dev.error() == kv.KV_ERR_INVALID_ARG
    assert int(b.dev.ctl[kv.KV_CTL_APPEND_STOP].item()) == 2
    b.assert_state_equal()


def test_handoff_bad_source_page_id():
    import paged_fp8_kv_append_gb300 as kv

    w = _workload(0, 4861)
    ks, vs = _rows(w, w.lens)
    src, spt, ssl = _source(w, ks, vs)
    spt[3, 1] = w.num_pages + 7
    b = Both(w, 0)
    b.dev.append_from_pool(w.B, src, spt, ssl, b.pt_d, b.et_d, b.sl_d)
    torch.cuda.synchronize()
    assert b.dev.error() == kv.KV_ERR_BAD_PAGE_ID


def test_handoff_full_gqa_batch_equals_append():
    """The whole GQA batch (32 requests, 4k-32k tokens, per-channel scales):
    the handoff from a bf16 pool writes exactly what kv_append_quantize of the
    same rows writes (same free list and tags), codes, scales and bookkeeping
    alike."""
    import paged_fp8_kv_append_gb300 as kv

    w = wl.gqa_batch()
    ks, vs = _rows(w, w.lens)
    src, spt, ssl = _source(w, ks, vs, check=False)
    mk = lambda: kv.KVPool(w.num_pages, 16, 8, 128, 128, dtype=0, device="cuda",  # noqa: E731
                           tags=wl.initial_tags(w), free_list=wl.free_list(w))
    tabs = lambda: (torch.full((w.B, w.max_pages), -1, dtype=torch.int32, device="cuda"),  # noqa: E731
                    torch.zeros((w.B, w.max_pages), dtype=torch.int32, device="cuda"),
                    torch.zeros(w.B, dtype=torch.int32, device="cuda"))
    a, (apt, aet, asl) = mk(), tabs()
    ind = torch.from_numpy(np.concatenate([[0], np.cumsum(w.lens)]).astype(np.int32)).cuda()
    a.append(w.B, torch.cat(ks), torch.cat(vs), ind, int(w.lens.max()), apt, aet, asl)
    del ks, vs
    h, (hpt, het, hsl) = mk(), tabs()
    h.append_from_pool(w.B, src, spt, ssl, hpt, het, hsl)
    torch.cuda.synchronize()
    assert a.error() == 0 and h.error() == 0
    for x, y in ((apt, hpt), (aet, het), (asl, hsl), (a.tags, h.tags), (a.ctl, h.ctl),
                 (a.k_scale, h.k_scale), (a.v_scale, h.v_scale), (a.k_cache, h.k_cache),
                 (a.v_cache, h.v_cache)):
        assert torch.equal(x, y)


def test_handoff_full_latent_workload_equals_append():
    """The whole latent workload (64 requests, 8k-64k rows of 576 values,
    page 64): the handoff from a bf16 latent pool writes exactly what
    kv_append_quantize of the same rows writes (same free list and tags),
    codes, scales and bookkeeping alike."""
    import paged_fp8_kv_append_gb300 as kv

    w = wl.latent_verify()
    ks = [wl.kv_rows(w, r, 0, int(w.lens[r]), device="cuda")[0] for r in range(w.B)]
    src, spt, ssl = _source(w, ks, ks, check=False)
    mk = lambda: kv.KVPool(w.num_pages, 64, 1, 576, 512, dtype=0, layout=1,  # noqa: E731
                           device="cuda", tags=wl.initial_tags(w), free_list=wl.free_list(w))
    tabs = lambda: (torch.full((w.B, w.max_pages), -1, dtype=torch.int32, device="cuda"),  # noqa: E731
                    torch.zeros((w.B, w.max_pages), dtype=torch.int32, device="cuda"),
                    torch.zeros(w.B, dtype=torch.int32, device="cuda"))
    a, (apt, aet, asl) = mk(), tabs()
    ind = torch.from_numpy(np.concatenate([[0], np.cumsum(w.lens)]).astype(np.int32)).cuda()
    a.append(w.B, torch.cat(ks), None, ind, int(w.lens.max()), apt, aet, asl)
    del ks
    h, (hpt, het, hsl) = mk(), tabs()
    h.append_from_pool(w.B, src, spt, ssl, hpt, het, hsl)
    torch.cuda.synchronize()
    assert a.error() == 0 and h.error() == 0
    for x, y in ((apt, hpt), (aet, het), (asl, hsl), (a.tags, h.tags), (a.ctl, h.ctl),
                 (a.k_scale, h.k_scale), (a.k_cache, h.k_cache)):
        assert torch.equal(x, y)
