"""GPU parity: the CUDA library against the oracle on identical seeded inputs
(GQA layout).  Cache bytes, scales, tags, page tables, lengths, free head and
abort masks must be bit-exact; attention outputs must satisfy
|o - r| <= 2e-3 + 1e-2 |r| elementwise against the fp64 oracle computed from
the same dequantised values.  All calls go through the C ABI."""
import numpy as np
import pytest
import torch

import workloads as wl
from pathrun import Both, bf16_to_f64, close

pytestmark = pytest.mark.gpu


def _q(w, dev="cuda"):
    return wl.queries(w, device=dev)


def _check_out(out, ref, written, abort_h, sentinel=7.0):
    got = bf16_to_f64(out.cpu().view(torch.int16).numpy().view(np.uint16))
    for r in range(len(written)):
        if written[r]:
            ok, mabs, mrel, worst = close(got[r], ref[r])
            assert ok, f"request {r}: max abs {mabs:.3g}, max rel {mrel:.3g}, worst excess {worst:.3g}"
        else:
            assert np.all(got[r] == sentinel), f"request {r} must be left untouched"


@pytest.mark.parametrize("dtype", [0, 1])
def test_tiny_full_path(dtype):
    w = wl.tiny()
    b = Both(w, dtype)
    st, stop = b.fill()
    assert (st, stop) == (0, w.B)
    torch.cuda.synchronize()
    b.assert_state_equal()
    b.make_stale()
    m_d, m_h = b.verify()
    assert m_h.tolist() == [0, 0, 1, 0]
    assert np.array_equal(m_d.cpu().numpy(), m_h)
    out, ref, written = b.attn(_q(w), m_d, m_h)
    assert written.tolist() == [1, 1, 0, 1]
    _check_out(out, ref, written, m_h)
    assert b.dev.error() == 0


@pytest.mark.parametrize("dtype", [0, 1])
def test_phases_equal_single_call(dtype):
    w = wl.tiny(seed=77)
    b = Both(w, dtype)
    b.fill()
    q = _q(w)
    m = torch.zeros(w.B, dtype=torch.uint8, device="cuda")
    mh = np.zeros(w.B, np.uint8)
    o1, _, _ = b.attn(q, m, mh)
    o2, _, _ = b.attn(q, m, mh, phases=True)
    assert torch.equal(o1, o2)
    # the no-op tracker (NULL mask) equals an all-zero mask
    o3, ref, written = b.attn(q, None, None)
    assert torch.equal(o1, o3)
    _check_out(o3, ref, written, None)


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("Hq", [8, 24])
def test_nothing_to_attend(dtype, Hq):
    """Batches with no page to read: every request aborted (outputs left
    untouched), and every request empty (no visible position: zero rows, as
    the oracle gives).  The split grid then has no unit of work at all."""
    w = wl.tiny(seed=88)
    if Hq != w.num_q_heads:
        import dataclasses

        w = dataclasses.replace(w, num_q_heads=Hq)
    b = Both(w, dtype)
    assert b.fill()[0] == 0
    q = _q(w)
    m_h = np.ones(w.B, np.uint8)
    m_d = torch.from_numpy(m_h).cuda()
    out, ref, written = b.attn(q, m_d, m_h)
    assert not written.any() and b.dev.error() == 0
    _check_out(out, ref, written, m_h)
    # the same pool with every request cut back to length 0
    b.sl_h[:] = 0
    b.sl_d.zero_()
    out, ref, written = b.attn(q, None, None)
    assert written.all() and b.dev.error() == 0
    got = bf16_to_f64(out.cpu().view(torch.int16).numpy().view(np.uint16))
    assert np.all(got == 0.0) and np.all(ref == 0.0)


@pytest.mark.parametrize("dtype", [0, 1])
def test_ragged_lengths_and_single_token_appends(dtype):
    """Lengths that end mid-page, zero-length requests, then decode-style
    one-row appends into partly filled pages (frozen scales), several rounds."""
    rng = np.random.default_rng(5)
    lens = np.array([0, 1, 15, 16, 17, 33, 250, 1000, 4097, 31], np.int32)
    w = wl.Workload("ragged", 991, lens, 32, 4, 128, 128, 16, 1, 0, 2048, float(np.float32(0.088)),
                    steps=40)
    b = Both(w, dtype)
    assert b.fill()[0] == 0
    for step in range(3):
        ks, vs = [], []
        for r in range(w.B):
            k, v = wl.kv_rows(w, r, 100000 + int(b.sl_h[r]), 1, device="cuda", tag=step + 1)
            ks.append(k)
            vs.append(v)
        st, stop = b.append(ks, vs, np.ones(w.B, np.int64))
        assert (st, stop) == (0, w.B)
    torch.cuda.synchronize()
    b.assert_state_equal()
    m_d, m_h = b.verify()
    assert not m_h.any() and np.array_equal(m_d.cpu().numpy(), m_h)
    out, ref, written = b.attn(_q(w), m_d, m_h)
    _check_out(out, ref, written, m_h)


@pytest.mark.parametrize("T,Hq,Hkv", [(2, 8, 2), (4, 4, 2), (8, 8, 8), (1, 16, 16)])
def test_multi_token_causal_and_group_sizes(T, Hq, Hkv):
    lens = np.array([3, 9, 40, 129, 2, 1], np.int32)
    w = wl.Workload("causal", 313 + T, lens, Hq, Hkv, 128, 128, 16, T, 0, 256,
                    float(np.float32(1 / np.sqrt(128))))
    b = Both(w, 0)
    b.fill()
    out, ref, written = b.attn(_q(w), None, None)
    _check_out(out, ref, written, None)


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("mag", [1e-4, 3e3])
@pytest.mark.parametrize("T,Hq", [(2, 16), (1, 48), (4, 32), (4, 64)])
def test_kv_magnitude_extremes(dtype, mag, T, Hq):
    """K/V drawn at 1e-4 and 3e3: page scales far from 1 (about 1e-6 and 30)
    must not push the attention weights out of f16's normal range.  Outputs
    are compared relative to the magnitude (the absolute term of the bound
    would otherwise hide a tiny-scale error).  8, 12, 32 and 64 query rows
    per kv head (4 kv heads)."""
    lens = np.array([37, 300, 1000, 5], np.int32)
    w = wl.Workload("magnitude", 123, lens, Hq, 4, 128, 128, 16, T, 0, 256,
                    float(np.float32(1 / np.sqrt(128))), magnitude=mag)
    b = Both(w, dtype)
    assert b.fill()[0] == 0
    torch.cuda.synchronize()
    b.assert_state_equal()
    out, ref, written = b.attn(_q(w), None, None)
    assert written.all() and b.dev.error() == 0
    got = bf16_to_f64(out.cpu().view(torch.int16).numpy().view(np.uint16))
    for r in range(w.B):
        ok, mabs, mrel, _ = close(got[r] / mag, ref[r] / mag)
        assert ok, f"request {r}: max abs {mabs:.3g}, max rel {mrel:.3g} (relative to {mag})"


def test_bad_page_id_is_not_read():
    """A request whose page table holds an out-of-range id, with the no-op
    tracker: no output, KV_ERR_BAD_PAGE_ID, other requests unaffected."""
    w = wl.tiny(seed=91)
    b = Both(w, 0)
    b.fill()
    b.pt_h[1, 2] = 10 ** 9
    b.pt_d[1, 2] = 10 ** 9
    out, ref, written = b.attn(_q(w), None, None)
    assert written.tolist() == [1, 0, 1, 1]
    _check_out(out, ref, written, None)
    assert b.dev.error() == b.kv.KV_ERR_BAD_PAGE_ID
    # the tag check catches the same mapping and aborts exactly that request
    m_d, m_h = b.verify()
    assert m_h.tolist() == [0, 1, 0, 0] and np.array_equal(m_d.cpu().numpy(), m_h)


def test_out_of_pages_stops_at_request():
    lens = np.array([40, 100, 20], np.int32)
    w = wl.Workload("oop", 5, lens, 8, 2, 128, 128, 16, 1, 0, 9, 0.1)
    b = Both(w, 0, num_pages=9)  # needs 3 + 7 + 2 pages
    st, stop = b.fill()
    assert (st, stop) == (4, 1)
    torch.cuda.synchronize()
    assert int(b.dev.ctl[2].item()) == 1 and b.dev.error() == 4
    b.assert_state_equal()


def test_bf16_inputs_exhaustive_codes_scale_one():
    """With a page amax of exactly 448 the scale is 1.0 and the stored code is
    the hardware conversion of the input itself: every finite bf16 value of
    magnitude <= 448 is checked against the oracle's encoder."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = bf16_to_f64(bits)
    keep = bits[np.isfinite(vals) & (np.abs(vals) <= 448.0)]
    D, P = 128, 16
    per_row = D - 1
    nrows = -(-len(keep) // per_row)
    rows = np.zeros((nrows, D), np.uint16)
    flat = np.zeros(nrows * per_row, np.uint16)
    flat[: len(keep)] = keep
    rows[:, :per_row] = flat.reshape(nrows, per_row)
    rows[:, per_row] = np.uint16(0x43E0)  # bf16 448.0 in every row -> amax 448 in every page
    nrows_p = -(-nrows // P) * P
    pad = np.zeros((nrows_p - nrows, D), np.uint16)
    pad[:, per_row] = np.uint16(0x43E0)
    rows = np.concatenate([rows, pad])
    lens = np.array([rows.shape[0]], np.int32)
    w = wl.Workload("codes", 1, lens, 1, 1, D, D, P, 1, 0, rows.shape[0] // P + 2, 1.0)
    b = Both(w, 0)
    t = torch.from_numpy(rows.view(np.int16)).view(torch.bfloat16).reshape(-1, 1, D).cuda()
    st, _ = b.append([t], [t], [rows.shape[0]])
    assert st == 0
    torch.cuda.synchronize()
    assert np.all(b.ref.k_scale[b.pt_h[0, : rows.shape[0] // P], 0] == 1.0)
    b.assert_state_equal()


@pytest.mark.parametrize("bad_at", [None, 0.7])
def test_append_many_requests_and_a_bad_free_list_entry(bad_at):
    """1500 requests (two chunks of the planner), short ragged lengths; with
    bad_at, a free-list entry 70% of the way in is not a page id: the call
    stops at the request that would pop it, earlier ones are served, and the
    pool state matches the oracle bit for bit."""
    rng = np.random.default_rng(17)
    lens = rng.integers(0, 41, 1500).astype(np.int32)
    need = int((-(-lens.astype(np.int64) // 16)).sum())
    w = wl.Workload("many", 123, lens, 4, 2, 128, 128, 16, 1, 0, need + 50,
                    float(np.float32(0.088)))
    free = wl.free_list(w).copy()
    if bad_at is not None:
        free[int(bad_at * need)] = -7
    b = Both(w, 0, free=free)
    st, stop = b.fill()
    torch.cuda.synchronize()
    if bad_at is None:
        assert (st, stop) == (0, w.B) and b.dev.error() == 0
    else:
        assert st == b.kv.KV_ERR_BAD_PAGE_ID and 0 < stop < w.B
        assert b.dev.error() == b.kv.KV_ERR_BAD_PAGE_ID
        assert int(b.dev.ctl[2].item()) == stop
    b.assert_state_equal()


# (T, Hq, Hkv): query rows per kv head R = T * Hq / Hkv beyond one block of 8 --
# GLM-class groups (96 q / 8 kv heads), speculative tokens on G = 8 and G = 16
# models, 64 query heads on one kv head, and ragged last blocks (R = 18, 25,
# 33, 40: row blocks padded where the consumer warps would not divide)
@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("T,Hq,Hkv", [(1, 96, 8), (2, 16, 2), (4, 16, 2), (3, 24, 4),
                                      (1, 32, 1), (5, 10, 2), (1, 64, 1), (4, 64, 4),
                                      (3, 44, 4), (2, 40, 2)])
def test_more_than_eight_rows_per_kv_head(dtype, T, Hq, Hkv):
    """More than 8 query rows per kv head: each (kv head, block of 16 rows)
    pair is served by its own consumer warp over the kv head's K/V tiles
    (e4m3 and bf16)."""
    lens = np.array([3, 9, 40, 129, 2, 1, 300], np.int32)
    w = wl.Workload("rows", 917 + T + Hq, lens, Hq, Hkv, 128, 128, 16, T, 0, 320,
                    float(np.float32(1 / np.sqrt(128))))
    b = Both(w, dtype)
    assert b.fill()[0] == 0
    out, ref, written = b.attn(_q(w), None, None)
    assert b.dev.error() == 0
    _check_out(out, ref, written, None)
