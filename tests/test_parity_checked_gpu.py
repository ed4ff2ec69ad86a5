"""GPU parity of paged_decode_attn_checked, decode attention with the page-tag
check fused into the page reads ("Smaller, faster, safer: running Kimi and
GLM at scale", section "Protecting a shared KV cache": a request whose
recorded (page, tag) list disagrees with the physical tags is aborted and
returns no data).  Its abort mask must equal the oracle's tag check bit for
bit; non-aborted outputs must match the oracle's attention within
|o - r| <= 2e-3 + 1e-2 |r|; aborted requests' rows stay untouched.  Also the
batch plan on both sides of the split kernel's own-plan limit (1023
requests), with the separate check and the fused one."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from pathrun import Both, bf16_to_f64, close

pytestmark = pytest.mark.gpu


def _checked(b, q, sentinel=7.0):
    w = b.w
    out = torch.full((w.B, w.q_tokens, w.num_q_heads, w.head_dim_v), sentinel,
                     dtype=torch.bfloat16, device="cuda")
    mask = torch.full((w.B,), 0xEE, dtype=torch.uint8, device="cuda")
    ws = torch.empty(b.dev.workspace_size(w.B, w.num_q_heads, w.q_tokens), dtype=torch.uint8,
                     device="cuda")
    b.kv.paged_decode_attn_checked(b.dev.handle, w.B, w.num_q_heads, w.q_tokens, q, b.pt_d,
                                   b.et_d, b.sl_d, w.sm_scale, out, mask, ws)
    return out, mask


def _check(out, ref, written, sentinel=7.0):
    got = bf16_to_f64(out.cpu().view(torch.int16).numpy().view(np.uint16))
    for r in range(len(written)):
        if written[r]:
            ok, mabs, mrel, _ = close(got[r], ref[r])
            assert ok, (r, mabs, mrel)
        else:
            assert np.all(got[r] == sentinel), f"request {r} must be left untouched"


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("Hq", [8, 24])
def test_checked_stale_tag(dtype, Hq):
    """4 requests (8 or 12 query rows per kv head), request 2 with one stale
    expected tag: mask [0, 0, 1, 0]; the others attend."""
    w = dataclasses.replace(wl.tiny(seed=4101 + Hq), num_q_heads=Hq)
    b = Both(w, dtype)
    assert b.fill()[0] == 0
    b.make_stale()
    m_h = oracle.verify(b.ref.num_pages, w.page_size, b.ref.tags, b.pt_h, b.et_h, b.sl_h)
    assert m_h.tolist() == [0, 0, 1, 0]
    q = wl.queries(w, device="cuda")
    out, mask = _checked(b, q)
    assert np.array_equal(mask.cpu().numpy(), m_h)
    ref, written = oracle.attn(b.ref, wl.bits_u16(q), b.pt_h, b.sl_h, m_h, w.sm_scale, Hq, 1)
    _check(out, ref, written)
    assert b.dev.error() == 0


@pytest.mark.parametrize("dtype", [0, 1])
def test_checked_page_id_out_of_range(dtype):
    """A page-table entry outside the pool aborts its request (as the tag
    check decides it) and reports KV_ERR_BAD_PAGE_ID; no page of the pool is
    misread."""
    w = wl.tiny(seed=4202)
    b = Both(w, dtype)
    assert b.fill()[0] == 0
    b.pt_h[1, 2] = w.num_pages + 3
    b.pt_d.copy_(torch.from_numpy(b.pt_h))
    m_h = oracle.verify(b.ref.num_pages, w.page_size, b.ref.tags, b.pt_h, b.et_h, b.sl_h)
    assert m_h.tolist() == [0, 1, 0, 0]
    q = wl.queries(w, device="cuda")
    out, mask = _checked(b, q)
    assert np.array_equal(mask.cpu().numpy(), m_h)
    ref, written = oracle.attn(b.ref, wl.bits_u16(q), b.pt_h, b.sl_h, m_h, w.sm_scale, 8, 1)
    _check(out, ref, written)
    assert b.dev.error() == b.kv.KV_ERR_BAD_PAGE_ID


def test_checked_invalid_length():
    """A length its page table cannot hold aborts that request and reports
    KV_ERR_INVALID_ARG."""
    w = wl.tiny(seed=4303)
    b = Both(w, 0)
    assert b.fill()[0] == 0
    b.sl_h[3] = w.max_pages * w.page_size + 5
    b.sl_d.copy_(torch.from_numpy(b.sl_h))
    m_h = oracle.verify(b.ref.num_pages, w.page_size, b.ref.tags, b.pt_h, b.et_h, b.sl_h)
    assert m_h.tolist() == [0, 0, 0, 1]
    q = wl.queries(w, device="cuda")
    out, mask = _checked(b, q)
    assert np.array_equal(mask.cpu().numpy(), m_h)
    ref, written = oracle.attn(b.ref, wl.bits_u16(q), b.pt_h, b.sl_h, m_h, w.sm_scale, 8, 1)
    _check(out, ref, written)
    assert b.dev.error() == b.kv.KV_ERR_INVALID_ARG


def test_checked_latent_stale_tag():
    """The latent (tensor-core) layout: 4 draft tokens x 16 heads, one stale
    tag in request 1."""
    lens = np.array([37, 300, 64, 1000], np.int32)
    w = wl.Workload("chk_lat", 4404, lens, 16, 1, 576, 512, 64, 4, 1, 64,
                    float(np.float32(1 / np.sqrt(576))), stale=[1])
    b = Both(w, 0)
    assert b.fill()[0] == 0
    b.make_stale()
    m_h = oracle.verify(b.ref.num_pages, w.page_size, b.ref.tags, b.pt_h, b.et_h, b.sl_h)
    assert m_h.tolist() == [0, 1, 0, 0]
    q = wl.queries(w, device="cuda")
    out, mask = _checked(b, q)
    assert np.array_equal(mask.cpu().numpy(), m_h)
    ref, written = oracle.attn(b.ref, wl.bits_u16(q), b.pt_h, b.sl_h, m_h, w.sm_scale, 16, 4)
    _check(out, ref, written)
    assert b.dev.error() == 0


@pytest.mark.parametrize("B", [1023, 1024, 1100])
@pytest.mark.parametrize("dtype", [0, 1])
def test_many_requests_plan(B, dtype):
    """Batches around the split kernel's own-plan limit (it plans up to 1023
    requests itself; larger batches take the plan kernel): every request of
    the separate check + attention and of the fused check is compared with
    the oracle; 1% of the requests carry a stale tag."""
    rng = np.random.default_rng(B + 10 * dtype)
    lens = rng.integers(1, 48, size=B).astype(np.int32)
    need = int((-(-lens.astype(np.int64) // 16)).sum())
    stale = sorted(rng.choice(B, size=max(1, B // 100), replace=False).tolist())
    w = wl.Workload(f"many{B}", 4500 + B, lens, 8, 2, 128, 128, 16, 1, 0, int(need * 1.1) + 16,
                    float(np.float32(1 / np.sqrt(128))), stale=stale)
    b = Both(w, dtype)
    assert b.fill()[0] == 0
    b.make_stale()
    m_d, m_h = b.verify()
    assert sorted(np.flatnonzero(m_h).tolist()) == stale
    assert np.array_equal(m_d.cpu().numpy(), m_h)
    q = wl.queries(w, device="cuda")
    out, ref, written = b.attn(q, m_d, m_h)
    _check(out, ref, written)
    out2, mask2 = _checked(b, q)
    assert np.array_equal(mask2.cpu().numpy(), m_h)
    _check(out2, ref, written)
    assert b.dev.error() == 0
