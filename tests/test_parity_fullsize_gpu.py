"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times.  Every request's bookkeeping (page tables, expected tags,
tags, lengths, free head, abort masks) is compared bit-exactly with the
oracle; cache bytes, scales and attention outputs are compared for sampled
(request, kv head) pairs, the oracle running a one-kv-head pool fed the same
rows in the same calls."""
import numpy as np
import pytest
import torch

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
    check and attention; the stale requests abort and are left untouched."""
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
    assert fs.attn_check(wl.queries(w, device="cuda"), m_d, m_h) == len(picks) * w.num_kv_heads
    assert fs.dev.error() == 0
