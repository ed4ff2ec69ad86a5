"""Bulk appends at the batch-size boundary of the persistent append kernels:
up to 16,384 requests a call, every CTA holds the per-request work prefix in
shared memory (64 KB at the limit); above it the call takes the compact
per-(request, page, head) kernel.  Both sides of the boundary must leave the
pool bit-identical to the oracle's append ("Smaller, faster, safer: running
Kimi and GLM at scale", section "Quantizing the KV cache": rows are
quantised to e4m3 as they are written into the paged cache)."""
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
