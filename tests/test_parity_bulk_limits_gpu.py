"""Limits.  Bulk appends at the batch-size boundary of the persistent append kernels:
up to 16,384 requests a call, every CTA holds the per-request work prefix in
shared memory (64 KB at the limit); above it the call takes the compact
per-(request, page, head) kernel.  Both sides of the boundary must leave the
pool bit-identical to the oracle's append ("Smaller, faster, safer: running
Kimi and GLM at scale", section "Quantizing the KV cache": rows are
quantised to e4m3 as they are written into the paged cache).  And an
attention batch too large for the plan's 32-bit prefix is refused."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from pathrun import Both

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B", [16384, 16385])
@pytest.mark.parametrize("dtype", [0, 1])
def test_bulk_append_batch_limit(B, dtype):
    rng = np.random.default_rng(B + dtype)
    P, H, D = 16, 1, 128
    counts = rng.integers(2 * P, 2 * P + 9, B).astype(np.int64)
    counts[rng.choice(B, B // 16, replace=False)] = 0        # empty slots append nothing
    counts[0] = 2 * P                                        # the call takes the bulk path
    more = rng.integers(2 * P, 3 * P, B).astype(np.int64)    # the second call's rows
    more[counts == 0] = 0
    first = int((-(-counts // P)).sum())
    second = int((-(-(counts + more) // P)).sum()) - first
    npg = first + second // 2  # the second call runs out of pages half way
    w = wl.Workload("limits", 7 + B, counts.astype(np.int32), 8, H, D, D, P, 1, 0, npg,
                    float(np.float32(1 / np.sqrt(D))), steps=3 * P)
    b = Both(w, dtype)
    g = torch.Generator(device="cuda").manual_seed(int(B) * 3 + dtype)
    n = int(counts.sum())
    k = torch.randn((n, H, D), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((n, H, D), generator=g, device="cuda").to(torch.bfloat16)
    ind = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    b.dev.append(B, k, v, torch.from_numpy(ind).cuda(), int(counts.max()), b.pt_d, b.et_d,
                 b.sl_d)
    st, stop = oracle.append(b.ref, wl.bits_u16(k), wl.bits_u16(v), ind, int(counts.max()),
                             b.pt_h, b.et_h, b.sl_h)
    torch.cuda.synchronize()
    assert (st, stop) == (0, B)
    assert b.dev.error() == 0
    b.assert_state_equal()
    # a second call writes into the partly filled last pages and pops new
    # ones until the free list runs out
    n2 = int(more.sum())
    k2 = torch.randn((n2, H, D), generator=g, device="cuda").to(torch.bfloat16)
    v2 = torch.randn((n2, H, D), generator=g, device="cuda").to(torch.bfloat16)
    ind2 = np.concatenate([[0], np.cumsum(more)]).astype(np.int32)
    st, stop = oracle.append(b.ref, wl.bits_u16(k2), wl.bits_u16(v2), ind2, int(more.max()),
                             b.pt_h, b.et_h, b.sl_h)
    b.dev.append(B, k2, v2, torch.from_numpy(ind2).cuda(), int(more.max()), b.pt_d, b.et_d,
                 b.sl_d)
    torch.cuda.synchronize()
    # both sides stop at the same request when the pool runs out of pages
    assert st == oracle.ERR_OUT_OF_PAGES and b.dev.error() == st
    assert 0 < stop < B and stop == int(b.dev.ctl[b.kv.KV_CTL_APPEND_STOP].item())
    b.assert_state_equal()


def test_attention_refuses_a_batch_too_large_to_plan():
    """Lengths no pool can back -- two requests of 2^31 - 1 tokens, 2^28 page
    units in all -- would overflow the plan's 32-bit prefix: the plan refuses
    the batch with KV_ERR_INVALID_ARG, reads no page and writes no output.
    (Called through the C ABI directly, which takes the page-table width as
    an argument; the refused batch reads none of it.)"""
    import paged_fp8_kv_append_gb300 as kv

    pool = kv.KVPool(64, 16, 2, 128, 128, dtype=0, device="cuda")
    B, Hq = 2, 8
    mp = (2 ** 31 - 1 + 15) // 16
    sl = torch.full((B,), 2 ** 31 - 1, dtype=torch.int32, device="cuda")
    pt = torch.zeros((B, 1), dtype=torch.int32, device="cuda")
    q = torch.zeros((B, 1, Hq, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.full((B, 1, Hq, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(pool.workspace_size(B, Hq, 1), dtype=torch.uint8, device="cuda")
    st = kv._lib.paged_decode_attn(pool.handle, torch.cuda.current_stream().cuda_stream, B, Hq,
                                   1, q.data_ptr(), pt.data_ptr(), mp, sl.data_ptr(), None,
                                   0.088, out.data_ptr(), ws.data_ptr(), ws.numel())
    assert st == kv.KV_OK
    torch.cuda.synchronize()
    assert pool.error() == kv.KV_ERR_INVALID_ARG
    assert torch.all(out == 7.0)


def test_append_refuses_a_length_past_int32():
    """An append that would take a request past 2^31 - 1 tokens is refused
    with KV_ERR_INVALID_ARG although the declared page-table width could hold
    it, as the oracle does; nothing changes.  (A page-aligned length and an
    exhausted free list: no page-table entry is touched whichever check
    fires.  Called through the C ABI, which takes the width as an argument.)"""
    import paged_fp8_kv_append_gb300 as kv

    pool = kv.KVPool(8, 16, 1, 128, 128, dtype=0, device="cuda")
    pool.ctl[kv.KV_CTL_FREE_HEAD] = 8  # every page handed out
    mp = 2 ** 27 + 1
    sl = torch.tensor([2 ** 31 - 16], dtype=torch.int32, device="cuda")
    pt = torch.full((1, 4), -1, dtype=torch.int32, device="cuda")
    et = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    k = torch.zeros((16, 1, 128), dtype=torch.bfloat16, device="cuda")
    ind = torch.tensor([0, 16], dtype=torch.int32, device="cuda")
    st = kv._lib.kv_append_quantize(pool.handle, torch.cuda.current_stream().cuda_stream, 1,
                                    k.data_ptr(), k.data_ptr(), ind.data_ptr(), 16, pt.data_ptr(),
                                    et.data_ptr(), mp, sl.data_ptr())
    assert st == kv.KV_OK
    torch.cuda.synchronize()
    assert pool.error() == kv.KV_ERR_INVALID_ARG
    assert int(pool.ctl[kv.KV_CTL_APPEND_STOP].item()) == 0
    assert int(pool.ctl[kv.KV_CTL_FREE_HEAD].item()) == 8
    assert sl.tolist() == [2 ** 31 - 16] and torch.all(pt == -1)
