"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times.  Every request's bookkeeping (page tables, expected tags,
tags, lengths, free head, abort masks) is compared bit-exactly with the
oracle; cache bytes, scales and attention outputs are compared for sampled
(request, kv head) pairs, the oracle running a one-kv-head pool fed the same
rows in the same calls."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from pathrun import FullSize

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [0, 1])
def test_gqa_batch_full_size_decode_steps(dtype):
    w = wl.gqa_batch(steps=3)
    rng = np.random.default_rng(1)
    sample = sorted(rng.choice(w.B, 3, replace=False).tolist()) + [int(np.argmax(w.lens))]
    fs = FullSize(w, dtype, sample=sample, heads=[0, 5])
    fs.fill()
    for s in range(2):
        st, stop = fs.step_append(s)
        assert (st, stop) == (0, w.B)
    torch.cuda.synchronize()
    fs.assert_bookkeeping()
    fs.assert_sampled_cache()
    m_d, m_h = fs.verify()
    assert not m_h.any() and np.array_equal(m_d.cpu().numpy(), m_h)
    assert fs.attn_check(wl.queries(w, device="cuda"), m_d, m_h) == len(sample) * 2
    assert fs.dev.error() == 0


def test_gqa_batch_full_size_every_request_and_head():
    """The whole GQA batch (32 requests, 8 kv heads, e4m3) after a decode
    step: cache bytes, scales and attention outputs of every request and
    every kv head against the oracle (one one-kv-head oracle pool per pair,
    256 in all)."""
    w = wl.gqa_batch(steps=2)
    fs = FullSize(w, 0, sample=list(range(w.B)), heads=list(range(w.num_kv_heads)))
    fs.fill()
    st, stop = fs.step_append(0)
    assert (st, stop) == (0, w.B)
    torch.cuda.synchronize()
    fs.assert_bookkeeping()
    fs.assert_sampled_cache()
    m_d, m_h = fs.verify()
    assert not m_h.any() and np.array_equal(m_d.cpu().numpy(), m_h)
    assert fs.attn_check(wl.queries(w, device="cuda"), m_d, m_h) == w.B * w.num_kv_heads
    assert fs.dev.error() == 0


@pytest.mark.parametrize("dtype", [0, 1])
def test_wide_group_full_size_sampled(dtype):
    """The GQA batch with 96 query heads on its 8 kv heads (12 query rows per
    kv head: the 16-row consumer warps), e4m3 and bf16, at full size after a
    decode step: bookkeeping of every request; cache bytes, scales and
    attention of a seeded 4 requests (the longest among them) on three kv
    heads."""
    import dataclasses

    w = dataclasses.replace(wl.gqa_batch(steps=2), num_q_heads=96)
    rng = np.random.default_rng(3)
    sample = sorted(set(rng.choice(w.B, 3, replace=False).tolist()) | {int(np.argmax(w.lens))})
    heads = [0, 4, 7]
    fs = FullSize(w, dtype, sample=sample, heads=heads)
    fs.fill()
    st, stop = fs.step_append(0)
    assert (st, stop) == (0, w.B)
    torch.cuda.synchronize()
    fs.assert_bookkeeping()
    fs.assert_sampled_cache()
    m_d, m_h = fs.verify()
    assert not m_h.any() and np.array_equal(m_d.cpu().numpy(), m_h)
    assert fs.attn_check(wl.queries(w, device="cuda"), m_d, m_h) == len(sample) * len(heads)
    assert fs.dev.error() == 0


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("B", [1, 8, 64])
def test_concurrency_128k_contexts(B, dtype):
    """Requests of 131,072 tokens, e4m3 and bf16 caches: at 1 and 8 requests
    every request and kv head is checked; at 64 a seeded 8 requests on three
    kv heads."""
    w = wl.concurrency(B)
    w.steps = 2
    if B <= 8:
        sample, heads = list(range(B)), list(range(w.num_kv_heads))
    else:
        sample = sorted(np.random.default_rng(B).choice(B, 8, replace=False).tolist())
        heads = [0, 3, 7]
    fs = FullSize(w, dtype, sample=sample, heads=heads)
    fs.fill(group=2)
    fs.step_append(0)
    torch.cuda.synchronize()
    fs.assert_bookkeeping()
    fs.assert_sampled_cache()
    assert fs.attn_check(wl.queries(w, device="cuda"), None, None) == len(sample) * len(heads)
    assert fs.dev.error() == 0


def test_skewed_stress_steps_with_stale_tags():
    """256 requests, lognormal contexts up to 256k; every step appends one
    token per request (pages come off a shuffled free list), then the tag
    check and attention; the stale requests abort and are left untouched.
    The last step's attention runs twice: after the separate check, and with
    the check fused into the page reads (paged_decode_attn_checked)."""
    w = wl.skewed(steps=4)
    rng = np.random.default_rng(5)
    live = [r for r in range(w.B) if r not in w.stale]
    # a seeded 16 non-aborted requests (the longest among them) on every kv
    # head, and the stale ones
    picks = sorted(set(rng.choice(live, 15, replace=False).tolist()) | {int(np.argmax(w.lens))})
    while len(picks) < 16:
        picks = sorted(set(picks) | {int(rng.choice(live))})
    fs = FullSize(w, 0, sample=sorted(set(picks) | set(w.stale)),
                  heads=list(range(w.num_kv_heads)))
    fs.fill(group=16)
    fs.make_stale()
    for s in range(3):
        st, stop = fs.step_append(s)
        assert (st, stop) == (0, w.B)
        m_d, m_h = fs.verify()
        assert np.array_equal(m_d.cpu().numpy(), m_h)
        assert sorted(np.nonzero(m_h)[0].tolist()) == sorted(w.stale)
        torch.cuda.synchronize()
        fs.assert_bookkeeping()  # every step
    fs.assert_sampled_cache()
    q = wl.queries(w, device="cuda")
    assert fs.attn_check(q, m_d, m_h) == len(picks) * w.num_kv_heads
    # the same step's attention with the check fused into its page reads:
    # the same abort mask, the same outputs, the stale requests untouched
    assert fs.attn_check(q, None, m_h, fused=True) == len(picks) * w.num_kv_heads
    assert fs.dev.error() == 0


def test_one_call_step_at_the_headline_size():
    """kv_decode_step -- tag check, append of one token per request, split-K
    attention and combine in one call, as the benchmark's end-to-end line
    runs it -- on 64 requests of 131,072 tokens (e4m3): bookkeeping of every
    request and the abort mask bit-exact, cache bytes and attention output of
    two sampled (request, kv head) pairs against the oracle."""
    from pathrun import bf16_to_f64, close, gqa_oracle_attn

    w = wl.concurrency(64)
    w.steps = 2
    fs = FullSize(w, 0, sample=[0, 37], heads=[3])
    fs.fill(group=4)
    B, dev = w.B, fs.dev
    k, v = wl.step_rows(w, 0, device="cuda")
    q = wl.queries(w, device="cuda")
    ones = np.ones(B, np.int64)
    ind = np.concatenate([[0], np.cumsum(ones)]).astype(np.int32)
    out = torch.full((B, w.q_tokens, w.num_q_heads, w.head_dim_v), 7.0, dtype=torch.bfloat16,
                     device="cuda")
    mask = torch.full((B,), 0xEE, dtype=torch.uint8, device="cuda")
    ws = torch.empty(dev.step_workspace_size(B, w.num_q_heads, w.q_tokens), dtype=torch.uint8,
                     device="cuda")
    dev.step(B, w.num_q_heads, w.q_tokens, None, k.contiguous(), v.contiguous(),
             torch.from_numpy(ind).cuda(), 1, fs.pt_d, fs.et_d, fs.sl_d, q, w.sm_scale, out,
             mask, 0, ws)
    # the oracle's side of the same step: every tag valid, so the check aborts
    # nothing and the append serves every request
    m_h = oracle.verify(fs.bk.num_pages, w.page_size, fs.bk.tags, fs.pt_h, fs.et_h, fs.sl_h)
    assert not m_h.any()
    st, stop = oracle.alloc(fs.bk, ind, 1, fs.pt_h, fs.et_h, fs.sl_h)
    assert (st, stop) == (0, B)
    for (r, h), (pool, pt, et, sl) in fs.twins.items():
        s2, _ = oracle.append(pool, wl.bits_u16(k[r:r + 1, h:h + 1, :]),
                              wl.bits_u16(v[r:r + 1, h:h + 1, :]), np.array([0, 1], np.int32),
                              1, pt, et, sl)
        assert s2 == 0
    torch.cuda.synchronize()
    assert dev.error() == 0
    assert np.array_equal(mask.cpu().numpy(), m_h)
    fs.assert_bookkeeping()
    fs.assert_sampled_cache()
    got = bf16_to_f64(out.cpu().view(torch.int16).numpy().view(np.uint16))
    G = w.num_q_heads // w.num_kv_heads
    for (r, h), (pool, pt, et, sl) in fs.twins.items():
        qs = wl.bits_u16(q[r:r + 1, :, h * G:(h + 1) * G, :].cpu())
        ref = gqa_oracle_attn((pool, qs, pt, sl, w.sm_scale, G, w.q_tokens))
        ok, mabs, mrel, _ = close(got[r, :, h * G:(h + 1) * G], ref)
        assert ok, (r, h, mabs, mrel)
