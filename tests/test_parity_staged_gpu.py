"""GPU parity of the bulk append's staged kernels over page shapes.

A bulk append (at least two pages' worth of rows per call, at most 4096
requests) runs one CTA per SM: a producer warp bulk-copies each page's K rows
and V rows (latent layout: its rows) into shared-memory stages and consumer
warps quantise or copy the page from there ("Smaller, faster, safer: running Kimi and GLM at
scale", section "Quantizing the KV cache": the cache is written as FP8
e4m3, or kept as BF16).  Two calls per case: the first fills every request
from empty (fresh pages, ragged last pages), the second appends into the
partly filled last pages (the page's existing scale, its tag checked) and
pops new ones.  After each call the whole pool -- codes or bf16 bits,
scales, tags, page tables, expected tags, lengths, free-list head -- must
equal the oracle's bit for bit.  GQA shapes: the 16-row, 128-wide pages
(whose partly filled V tiles are written element by element) and others
(which assemble them in a per-warp shared tile), and K and V of different
widths.  Latent shapes: the 64-row, 576-wide pages (12 chunks per consumer
thread, every one used) and smaller ones."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from pathrun import Both

pytestmark = pytest.mark.gpu

SHAPES = [  # page size, kv heads, K width, V width
    (16, 8, 128, 128),
    (16, 3, 128, 128),
    (32, 2, 64, 64),
    (8, 4, 256, 256),
    (16, 2, 64, 128),
    (16, 1, 32, 32),
]


LATENT_SHAPES = [  # page size, K width (the row), V width (its leading part)
    (64, 576, 512),
    (32, 256, 256),
    (16, 64, 64),
]


def _rows(g, n, H, D, mags):
    """bf16 rows [n][H][D] ([n][D] when H is None); each row drawn at one of a
    few magnitudes, so that pages get different scales."""
    shape = (n, D) if H is None else (n, H, D)
    x = torch.randn(shape, generator=g, device="cuda")
    pick = torch.randint(0, len(mags), (n,) + (1,) * (len(shape) - 1), generator=g,
                         device="cuda")
    return (x * torch.tensor(mags, device="cuda")[pick]).to(torch.bfloat16)


def _counts(rng, P, B):
    first = rng.integers(2 * P, 9 * P, B)
    first[rng.choice(B, 4, replace=False)] = 0                 # no rows in the first call
    exact = rng.choice(np.flatnonzero(first), 5, replace=False)
    first[exact] = (first[exact] // P) * P                     # whole last pages
    second = rng.integers(2 * P, 5 * P, B)
    second[rng.choice(B, 3, replace=False)] = 0
    return first, second


def _two_calls(b, first, second, mode, rows):
    B = b.w.B
    # in requantising mode the second call's rows are larger, so the partly
    # filled pages take a larger scale and their old codes are re-encoded
    for counts, mags in ((first, [0.25, 1.0, 8.0]), (second, [0.5, 4.0, 64.0] if mode else
                                                      [0.25, 1.0, 8.0])):
        ks, vs = rows(counts, mags)
        st, stop = b.append(ks, vs, counts)
        assert (st, stop) == (0, B)
        torch.cuda.synchronize()
        assert b.dev.error() == 0
        b.assert_state_equal()


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("dtype,mode", [(0, 0), (1, 0), (0, 1)])
def test_staged_bulk_append_two_calls(shape, dtype, mode):
    P, H, Dk, Dv = shape
    rng = np.random.default_rng(P * 100003 + H * 1009 + Dk * 31 + Dv * 7 + dtype * 3 + mode)
    B = 37
    first, second = _counts(rng, P, B)
    total = first + second
    need = int((-(-total // P)).sum()) + 8
    w = wl.Workload("staged", 8100 + P + H, total.astype(np.int32), H, H, Dk, Dv, P, 1, 0,
                    need, float(np.float32(1 / np.sqrt(Dk))))
    b = Both(w, dtype, scale_mode=mode)
    g = torch.Generator(device="cuda").manual_seed(int(rng.integers(0, 2 ** 31)))
    _two_calls(b, first, second, mode,
               lambda counts, mags: ([_rows(g, int(c), H, Dk, mags) for c in counts],
                                     [_rows(g, int(c), H, Dv, mags) for c in counts]))


@pytest.mark.parametrize("shape", LATENT_SHAPES)
@pytest.mark.parametrize("dtype,mode", [(0, 0), (1, 0), (0, 1)])
def test_staged_latent_bulk_append_two_calls(shape, dtype, mode):
    P, Dk, Dv = shape
    rng = np.random.default_rng(P * 7919 + Dk * 13 + dtype * 3 + mode)
    B = 29
    first, second = _counts(rng, P, B)
    total = first + second
    need = int((-(-total // P)).sum()) + 8
    w = wl.Workload("staged_lat", 8200 + P, total.astype(np.int32), 16, 1, Dk, Dv, P, 1, 1,
                    need, float(np.float32(1 / np.sqrt(Dk))))
    b = Both(w, dtype, scale_mode=mode)
    g = torch.Generator(device="cuda").manual_seed(int(rng.integers(0, 2 ** 31)))

    def rows(counts, mags):
        ks = [_rows(g, int(c), None, Dk, mags) for c in counts]
        return ks, ks

    _two_calls(b, first, second, mode, rows)


@pytest.mark.parametrize("layout", [0, 1])
def test_staged_and_register_kernels_agree_at_the_batch_limit(layout):
    """4096 requests take the staged kernels, 4097 the register-resident
    ones: the same rows appended from empty (the 4097th request empty) leave
    the same pool bit for bit, and both equal the oracle."""
    import paged_fp8_kv_append_gb300 as kv

    rng = np.random.default_rng(9100 + layout)
    B = 4096
    if layout == 0:
        P, H, Dk, Dv = 16, 1, 128, 128
    else:
        P, H, Dk, Dv = 64, 1, 64, 64
    counts = rng.integers(2 * P, 3 * P + 5, B)
    counts[rng.choice(B, 64, replace=False)] = 0
    need = int((-(-counts // P)).sum()) + 8
    g = torch.Generator(device="cuda").manual_seed(9100 + layout)
    n = int(counts.sum())
    if layout == 0:
        k = _rows(g, n, H, Dk, [0.25, 1.0, 8.0])
        v = _rows(g, n, H, Dv, [0.25, 1.0, 8.0])
    else:
        k = _rows(g, n, None, Dk, [0.25, 1.0, 8.0])
        v = None
    pools = []
    for Bc in (B, B + 1):
        cnt = np.concatenate([counts, np.zeros(Bc - B, np.int64)])
        w = wl.Workload("limit", 9100, cnt.astype(np.int32), H, H, Dk, Dv, P, 1, layout, need,
                        float(np.float32(1 / np.sqrt(Dk))))
        b = Both(w, 0)
        ind = np.concatenate([[0], np.cumsum(cnt)]).astype(np.int32)
        b.dev.append(Bc, k, v, torch.from_numpy(ind).cuda(), int(cnt.max()), b.pt_d, b.et_d,
                     b.sl_d)
        torch.cuda.synchronize()
        assert b.dev.error() == 0
        pools.append(b)
    a, c = pools
    assert torch.equal(a.dev.k_cache, c.dev.k_cache) and torch.equal(a.dev.k_scale, c.dev.k_scale)
    if layout == 0:
        assert torch.equal(a.dev.v_cache, c.dev.v_cache)
        assert torch.equal(a.dev.v_scale, c.dev.v_scale)
    assert torch.equal(a.pt_d, c.pt_d[:B]) and torch.equal(a.sl_d, c.sl_d[:B])
    # and the staged result is the oracle's
    ind = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    st, stop = oracle.append(a.ref, wl.bits_u16(k), None if v is None else wl.bits_u16(v), ind,
                             int(counts.max()), a.pt_h, a.et_h, a.sl_h)
    assert (st, stop) == (0, B)
    a.assert_state_equal()


@pytest.mark.parametrize("layout", [0, 1])
def test_staged_bulk_append_stops_at_a_stale_partial_page(layout):
    """A bulk second call in which request 5's partly filled last page carries
    a stale expected tag: the call serves requests 0-4, stops at 5 with
    KV_ERR_TAG_MISMATCH (its index in ctl[KV_CTL_APPEND_STOP]) and leaves
    request 5 and every later one untouched -- the same state as the oracle,
    bit for bit."""
    import paged_fp8_kv_append_gb300 as kv

    rng = np.random.default_rng(9300 + layout)
    B = 12
    if layout == 0:
        P, H, Dk, Dv = 16, 8, 128, 128
    else:
        P, H, Dk, Dv = 64, 1, 576, 512
    first = rng.integers(2 * P + 1, 5 * P, B)
    first[first % P == 0] += 3                     # every request ends in a partial page
    second = rng.integers(2 * P, 4 * P, B)
    total = first + second
    need = int((-(-total // P)).sum()) + 8
    w = wl.Workload("stale_partial", 9300, total.astype(np.int32), 8 if layout == 0 else 16,
                    H, Dk, Dv, P, 1, layout, need, float(np.float32(1 / np.sqrt(Dk))))
    b = Both(w, 0)
    g = torch.Generator(device="cuda").manual_seed(9300 + layout)

    def rows(counts):
        if layout == 0:
            return ([_rows(g, int(c), H, Dk, [1.0]) for c in counts],
                    [_rows(g, int(c), H, Dv, [1.0]) for c in counts])
        ks = [_rows(g, int(c), None, Dk, [1.0]) for c in counts]
        return ks, ks

    st, stop = b.append(*rows(first), first)
    assert (st, stop) == (0, B)
    r, j = 5, int(first[5] // P)                   # request 5's partly filled page
    b.et_h[r, j] = np.uint32(b.et_h[r, j]) - np.uint32(1)
    b.et_d.copy_(torch.from_numpy(b.et_h.view(np.int32)))
    st, stop = b.append(*rows(second), second)
    assert (st, stop) == (oracle.ERR_TAG_MISMATCH, 5)
    torch.cuda.synchronize()
    assert b.dev.error() == kv.KV_ERR_TAG_MISMATCH
    assert int(b.dev.ctl[kv.KV_CTL_APPEND_STOP].item()) == 5
    b.assert_state_equal()
