"""Continuous batching over fixed request slots ("Smaller, faster, safer:
running Kimi and GLM at scale", section "Protecting a shared KV cache": the
check stays on for every step while requests come and go).  A slot whose
length is 0 is empty: append writes nothing for it, the tag check reads no
page, attention reads nothing and writes a zero row.  Each round: finished
requests release their pages (their slots become empty), new requests join
empty slots with a bulk append of their prompt, then every slot takes a
decode step (append -> verify -> attention).  A request whose tag goes
stale is aborted by the check and removed the same way.  Pool state is
compared with the oracle bit for bit after every round, attention within
the usual bound."""
import numpy as np
import pytest
import torch

import workloads as wl
from pathrun import Both, bf16_to_f64, close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [0, 1])
def test_join_leave_abort_rounds(dtype):
    rng = np.random.default_rng(5 + dtype)
    S = 12  # slots
    lens = np.zeros(S, np.int32)
    w = wl.Workload("churn", 91 + dtype, lens, 16, 4, 128, 128, 16, 1, 0, 600,
                    float(np.float32(1 / np.sqrt(128))), steps=400)
    b = Both(w, dtype)
    active = set()
    tag = 0

    def rows(r, n):
        nonlocal tag
        tag += 1
        return wl.kv_rows(w, r, 300000 + int(b.sl_h[r]), n, device="cuda", tag=tag)

    def append(counts):
        ks, vs = [], []
        for r in range(S):
            k, v = rows(r, int(counts[r])) if counts[r] else (None, None)
            ks.append(k)
            vs.append(v)
        return b.append(ks, vs, counts)

    stale_round = 3
    for rnd in range(7):
        # leave: a few finished requests give their pages back
        if active:
            leave = rng.choice(sorted(active), size=min(2, len(active)), replace=False)
            mask = np.zeros(S, np.uint8)
            mask[leave] = 1
            assert b.release(mask) == 0
            active -= set(int(x) for x in leave)
        # join: new requests take empty slots with their prompts (bulk append)
        free = [r for r in range(S) if r not in active]
        join = rng.choice(free, size=min(3, len(free)), replace=False)
        counts = np.zeros(S, np.int64)
        counts[join] = rng.integers(1, 200, len(join))
        assert append(counts) == (0, S)
        active |= set(int(x) for x in join)
        torch.cuda.synchronize()
        b.assert_state_equal()
        if rnd == stale_round:  # one live request's mapping goes stale
            victim = sorted(active)[0]
            b.et_h[victim, 0] = np.uint32(b.et_h[victim, 0]) - np.uint32(1)
            b.et_d.copy_(torch.from_numpy(b.et_h.view(np.int32)))
        # decode step over every slot: empty slots append nothing
        counts = np.array([1 if r in active else 0 for r in range(S)], np.int64)
        assert append(counts) == (0, S)
        m_d, m_h = b.verify()
        assert np.array_equal(m_d.cpu().numpy(), m_h)
        assert set(np.flatnonzero(m_h).tolist()) <= active
        if rnd == stale_round:
            assert m_h[victim] == 1
        out, ref, written = b.attn(wl.queries(w, device="cuda", step=rnd), m_d, m_h)
        got = bf16_to_f64(out.cpu().view(torch.int16).numpy().view(np.uint16))
        for r in range(S):
            if written[r]:
                ok, mabs, mrel, _ = close(got[r], ref[r])
                assert ok, f"round {rnd} slot {r}: max abs {mabs:.3g} max rel {mrel:.3g}"
                if r not in active:
                    assert np.all(got[r] == 0)  # an empty slot's row is zero
        # aborted requests are removed like finished ones
        if m_h.any():
            assert b.release(m_h) == 0
            active -= set(np.flatnonzero(m_h).tolist())
        torch.cuda.synchronize()
        assert b.dev.error() == 0
        b.assert_state_equal()
