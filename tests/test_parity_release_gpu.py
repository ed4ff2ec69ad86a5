"""GPU parity of the page lifecycle: kv_release_pages, reallocation of the
released pages (tags bumped on re-pop), the stale mappings that then fail the
tag check, and append's tag check on a partly filled page ("Smaller, faster,
safer: running Kimi and GLM at scale", section "Protecting a shared KV
cache").  Pool state is compared bit-exactly with the oracle, free list and
free head included; attention after reuse within the usual tolerance."""
import numpy as np
import pytest
import torch

import workloads as wl
from pathrun import Both, bf16_to_f64, close

pytestmark = pytest.mark.gpu


def _w(lens, layout=0, seed=41):
    lens = np.array(lens, np.int32)
    if layout == 0:
        npg = int((-(-lens.astype(np.int64) // 16)).sum()) + 40
        return wl.Workload("lifecycle", seed, lens, 16, 4, 128, 128, 16, 1, 0, npg,
                           float(np.float32(1 / np.sqrt(128))), steps=1200)
    npg = int((-(-lens.astype(np.int64) // 64)).sum()) + 16
    return wl.Workload("lifecycle_latent", seed, lens, 16, 1, 576, 512, 64, 4, 1, npg,
                       float(np.float32(1 / np.sqrt(576))), steps=1200)


def _check_attn(b, q):
    out, ref, written = b.attn(q, None, None)
    got = bf16_to_f64(out.cpu().view(torch.int16).numpy().view(np.uint16))
    for r in range(b.w.B):
        if written[r]:
            ok, mabs, mrel, _ = close(got[r], ref[r])
            assert ok, f"request {r}: max abs {mabs:.3g} max rel {mrel:.3g}"


@pytest.mark.parametrize("dtype", [0, 1])
def test_release_reuse_and_stale_mappings(dtype):
    w = _w([37, 300, 64, 1000, 5, 129], seed=41 + dtype)
    b = Both(w, dtype)
    assert b.fill()[0] == 0
    old = (b.pt_h.copy(), b.et_h.copy(), b.sl_h.copy())
    mask = np.array([1, 0, 1, 0, 0, 1], np.uint8)
    assert b.release(mask) == 0
    torch.cuda.synchronize()
    assert b.dev.error() == 0
    b.assert_state_equal()
    assert b.sl_h.tolist() == [0, 300, 0, 1000, 5, 0]
    # the released requests start again; together they re-pop every released page
    news = np.array([200, 0, 90, 0, 0, 70], np.int64)
    ks, vs = [], []
    for r in range(w.B):
        k, v = wl.kv_rows(w, r, 0, int(news[r]), device="cuda", tag=7)
        ks.append(k)
        vs.append(v)
    assert b.append(ks, vs, news) == (0, w.B)
    torch.cuda.synchronize()
    assert b.dev.error() == 0
    b.assert_state_equal()
    # the mappings recorded before the release are stale now: tag check aborts them
    pt_o, et_o, sl_o = (torch.from_numpy(old[0]).cuda(), torch.from_numpy(old[1].view(np.int32))
                        .cuda(), torch.from_numpy(old[2]).cuda())
    m_d = torch.zeros(w.B, dtype=torch.uint8, device="cuda")
    b.dev.verify(w.B, pt_o, et_o, sl_o, m_d)
    import oracle
    m_h = oracle.verify(b.ref.num_pages, w.page_size, b.ref.tags, old[0], old[1], old[2])
    assert np.array_equal(m_d.cpu().numpy(), m_h)
    assert m_h.tolist() == mask.tolist()
    # the live mappings pass, and attention over the reused pages matches
    m_d, m_h = b.verify()
    assert not m_h.any() and np.array_equal(m_d.cpu().numpy(), m_h)
    _check_attn(b, wl.queries(w, device="cuda"))


def test_release_all_and_refill_latent():
    w = _w([700, 64, 130, 2], layout=1)
    b = Both(w, 0)
    assert b.fill()[0] == 0
    assert b.release(None) == 0
    torch.cuda.synchronize()
    b.assert_state_equal()
    assert int(b.dev.ctl[0].item()) == 0
    assert b.fill(lens=np.array([65, 500, 1, 64], np.int32), tag=3)[0] == 0
    torch.cuda.synchronize()
    b.assert_state_equal()
    _check_attn(b, wl.queries(w, device="cuda"))


@pytest.mark.parametrize("dtype", [0, 1])
def test_append_stops_at_a_reallocated_partial_page(dtype):
    w = _w([37, 300, 64, 1000, 5, 129], seed=43)
    b = Both(w, dtype)
    b.fill()
    torch.cuda.synchronize()
    # request 3's partly filled page (1000 = 62 * 16 + 8) changed hands
    p = int(b.pt_h[3, 1000 // 16])
    b.ref.tags[p] += np.uint32(1)
    b.dev.tags[p] += 1
    ks, vs = [], []
    for r in range(w.B):
        k, v = wl.kv_rows(w, r, int(b.sl_h[r]), 1, device="cuda", tag=9)
        ks.append(k)
        vs.append(v)
    st, stop = b.append(ks, vs, np.ones(w.B, np.int64))
    torch.cuda.synchronize()
    assert (st, stop) == (b.kv.KV_ERR_TAG_MISMATCH, 3)
    assert b.dev.error() == b.kv.KV_ERR_TAG_MISMATCH
    assert int(b.dev.ctl[2].item()) == 3
    b.assert_state_equal()  # requests 0..2 appended, 3..5 untouched


@pytest.mark.parametrize("dtype", [0, 1])
def test_append_stops_at_a_partial_page_popped_earlier_in_the_same_call(dtype):
    """A partly filled page listed free again and popped by an earlier request
    of the same call: the later request's check sees the bumped tag."""
    w = _w([37, 300, 64, 1000, 5, 129], seed=45)
    b = Both(w, dtype)
    b.fill()
    torch.cuda.synchronize()
    # request 3's partly filled page (1000 = 62 * 16 + 8) goes on top of the
    # free list; request 2 (64 rows: 4 full pages) pops it for its next row
    p = int(b.pt_h[3, 1000 // 16])
    head = int(b.ref.free_head[0])
    b.ref.free_list[head] = p
    b.dev.free_list[head] = p
    ks, vs = [], []
    for r in range(w.B):
        k, v = wl.kv_rows(w, r, int(b.sl_h[r]), 1, device="cuda", tag=11)
        ks.append(k)
        vs.append(v)
    st, stop = b.append(ks, vs, np.ones(w.B, np.int64))
    torch.cuda.synchronize()
    assert (st, stop) == (b.kv.KV_ERR_TAG_MISMATCH, 3)
    assert b.dev.error() == b.kv.KV_ERR_TAG_MISMATCH
    assert int(b.dev.ctl[2].item()) == 3
    assert int(b.pt_h[2, 64 // 16]) == p
    b.assert_state_equal()  # requests 0..2 appended (2 holds page p), 3..5 untouched


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("scale_mode", [0, 1])
def test_no_write_into_a_partial_page_a_later_request_of_the_call_pops(dtype, scale_mode):
    """A partly filled page listed free again and popped by a later request of
    the same call: the earlier request is served (its check comes first) but
    its row does not go into the page, which now holds the later request's
    rows and scale; the next check aborts the stale request."""
    if dtype == 1 and scale_mode == 1:
        pytest.skip("the re-quantising mode applies to e4m3 pools")
    w = _w([37, 300, 64, 1000, 5, 129], seed=46)
    b = Both(w, dtype, scale_mode=scale_mode)
    b.fill()
    torch.cuda.synchronize()
    # request 1's partly filled page (300 = 18 * 16 + 12) goes on top of the
    # free list; request 2 (64 rows: 4 full pages) pops it; request 3 joins
    # with 20 rows of which the first 8 fill its own partly filled page
    p = int(b.pt_h[1, 300 // 16])
    head = int(b.ref.free_head[0])
    b.ref.free_list[head] = p
    b.dev.free_list[head] = p
    counts = np.array([1, 1, 17, 20, 1, 1], np.int64)
    ks, vs = [], []
    for r in range(w.B):
        k, v = wl.kv_rows(w, r, int(b.sl_h[r]), int(counts[r]), device="cuda", tag=13)
        if r == 1:  # a row that would need a larger scale (exact: a power of two)
            k, v = (k.float() * 4).to(torch.bfloat16), (v.float() * 4).to(torch.bfloat16)
        ks.append(k)
        vs.append(v)
    st, stop = b.append(ks, vs, counts)
    torch.cuda.synchronize()
    assert (st, stop) == (0, w.B) and b.dev.error() == 0
    assert int(b.pt_h[2, 64 // 16]) == p
    b.assert_state_equal()  # cache bytes, scales and bookkeeping, bit-exact
    m_d, m_h = b.verify()
    assert np.array_equal(m_d.cpu().numpy(), m_h) and m_h.tolist() == [0, 1, 0, 0, 0, 0]
    q = wl.queries(w, device="cuda")
    out, ref, written = b.attn(q, m_d, m_h)
    got = bf16_to_f64(out.cpu().view(torch.int16).numpy().view(np.uint16))
    for r in range(w.B):
        if written[r]:
            ok, mabs, mrel, _ = close(got[r], ref[r])
            assert ok, f"request {r}: max abs {mabs:.3g} max rel {mrel:.3g}"


@pytest.mark.parametrize("scale_mode", [0, 1])
def test_no_write_into_a_partial_page_a_later_request_pops_latent(scale_mode):
    """The same on a latent pool (page 64, one scale per page): request 0's
    partly filled page (130 = 2 * 64 + 2) is popped by request 1 of the same
    call and holds only request 1's rows and scale afterwards."""
    w = _w([130, 64, 700, 2], layout=1, seed=47)
    b = Both(w, 0, scale_mode=scale_mode)
    b.fill()
    torch.cuda.synchronize()
    p = int(b.pt_h[0, 130 // 64])
    head = int(b.ref.free_head[0])
    b.ref.free_list[head] = p
    b.dev.free_list[head] = p
    counts = np.array([1, 70, 1, 1], np.int64)
    ks = []
    for r in range(w.B):
        k, _ = wl.kv_rows(w, r, int(b.sl_h[r]), int(counts[r]), device="cuda", tag=14)
        if r == 0:  # a row that would need a larger scale (exact: a power of two)
            k = (k.float() * 4).to(torch.bfloat16)
        ks.append(k)
    st, stop = b.append(ks, [None] * w.B, counts)
    torch.cuda.synchronize()
    assert (st, stop) == (0, w.B) and b.dev.error() == 0
    assert int(b.pt_h[1, 1]) == p
    b.assert_state_equal()
    m_d, m_h = b.verify()
    assert np.array_equal(m_d.cpu().numpy(), m_h) and m_h.tolist() == [1, 0, 0, 0]


def test_release_refused_when_more_than_handed_out():
    w = _w([37, 300, 64], seed=44)
    b = Both(w, 0)
    b.fill()
    torch.cuda.synchronize()
    head = int(b.ref.free_head[0])
    b.ref.free_head[0] = head - 2  # both sides believe fewer pages were handed out
    b.dev.ctl[0] = head - 2
    assert b.release(None) == b.kv.KV_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert b.dev.error() == b.kv.KV_ERR_INVALID_ARG
    b.assert_state_equal()  # nothing changed
