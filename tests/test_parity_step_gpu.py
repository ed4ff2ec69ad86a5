"""GPU parity of the continuous-batching step kv_decode_step ("Smaller,
faster, safer: running Kimi and GLM at scale", section "Protecting a shared
KV cache": the tag check is on for every step while requests join and
leave; a request whose pages were reallocated is aborted and returns no
data).  One call releases the leaving requests, checks the tags, appends
(joining requests' prompts, everyone else's new rows; aborted requests'
rows are dropped), attends, and removes the aborted requests.  The device
abort mask and pool state must equal the oracle's step bit for bit after
every step, attention within the usual bound."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from pathrun import Both, bf16_to_f64, close

pytestmark = pytest.mark.gpu

SENTINEL = 7.0


def _check_step(b, res, rnd, expect_status=0):
    st, m_d, m_h, out, ref, written = res
    torch.cuda.synchronize()
    assert st == expect_status, (rnd, st)
    assert b.dev.error() == expect_status, (rnd, b.kv.kv_status_string(b.dev.error()))
    assert np.array_equal(m_d.cpu().numpy(), m_h), (rnd, m_d.cpu().numpy(), m_h)
    b.assert_state_equal()
    got = bf16_to_f64(out.cpu().view(torch.int16).numpy().view(np.uint16))
    for r in range(b.w.B):
        if written[r]:
            ok, mabs, mrel, _ = close(got[r], ref[r])
            assert ok, f"step {rnd} slot {r}: max abs {mabs:.3g} max rel {mrel:.3g}"
        else:
            assert np.all(got[r] == SENTINEL), (rnd, r)


class _Rows:
    def __init__(self, b):
        self.b, self.tag = b, 0

    def __call__(self, counts):
        w, ks, vs = self.b.w, [], []
        for r in range(w.B):
            n = int(counts[r])
            if n == 0:
                ks.append(None)
                vs.append(None)
                continue
            self.tag += 1
            k, v = wl.kv_rows(w, r, 300000 + int(self.b.sl_h[r]), n, device="cuda", tag=self.tag)
            ks.append(k)
            vs.append(v)
        return ks, vs


@pytest.mark.parametrize("dtype", [0, 1])
def test_step_join_leave_abort(dtype):
    rng = np.random.default_rng(17 + dtype)
    S = 12
    w = wl.Workload("step", 171 + dtype, np.zeros(S, np.int32), 16, 4, 128, 128, 16, 1, 0, 700,
                    float(np.float32(1 / np.sqrt(128))), steps=600)
    b = Both(w, dtype)
    rows = _Rows(b)
    active = set()
    for rnd in range(8):
        leave = np.zeros(S, np.uint8)
        if len(active) >= 2:
            gone = rng.choice(sorted(active), size=2, replace=False)
            leave[gone] = 1
            active -= set(int(x) for x in gone)
        free = [r for r in range(S) if r not in active]
        join = rng.choice(free, size=min(3, len(free)), replace=False)
        counts = np.zeros(S, np.int64)
        counts[join] = rng.integers(1, 300, len(join))
        for r in active:
            counts[r] = 1
        victims = []
        if rnd in (2, 5) and active:
            # step 2 of the loop: a live request's partly filled last page went
            # stale (an append that wrote first would have hit it); step 5: an
            # inner page
            cand = sorted(active)
            part = [r for r in cand if b.sl_h[r] % 16 != 0 and b.sl_h[r] > 16]
            r = (part or cand)[0]
            j = int((b.sl_h[r] - 1) // 16) if rnd == 2 else 0
            b.et_h[r, j] = np.uint32(b.et_h[r, j]) - np.uint32(1)
            b.et_d.copy_(torch.from_numpy(b.et_h.view(np.int32)))
            victims.append(r)
        ks, vs = rows(counts)
        res = b.step(leave if leave.any() else None, ks, vs, counts,
                     wl.queries(w, device="cuda", step=rnd))
        _check_step(b, res, rnd)
        m_h = res[2]
        assert set(np.flatnonzero(m_h).tolist()) == set(victims)
        for r in victims:  # removed in the same call: the slot is empty again
            assert b.sl_h[r] == 0
        active |= set(int(x) for x in join)
        active -= set(victims)


def test_step_out_of_pages_then_recovers():
    """A join needing more pages than are free stops the append: that request
    and every later one are marked unserved, keep their state and attend
    nothing; after some requests leave, the next step serves everyone."""
    S = 6
    w = wl.Workload("step_oop", 33, np.zeros(S, np.int32), 16, 4, 128, 128, 16, 1, 0, 40,
                    float(np.float32(1 / np.sqrt(128))), steps=600)
    b = Both(w, 0)
    rows = _Rows(b)
    counts = np.array([100, 90, 0, 80, 0, 0])            # 7 + 6 + 5 = 18 pages
    ks, vs = rows(counts)
    _check_step(b, b.step(None, ks, vs, counts, wl.queries(w, device="cuda", step=0)), 0)
    counts = np.array([1, 1, 400, 1, 1, 0])              # slot 2 needs 25 pages; 22 are free
    ks, vs = rows(counts)
    res = b.step(None, ks, vs, counts, wl.queries(w, device="cuda", step=1))
    _check_step(b, res, 1, expect_status=b.kv.KV_ERR_OUT_OF_PAGES)
    assert res[2].tolist() == [0, 0, 2, 2, 2, 2]
    b.dev.ctl[b.kv.KV_CTL_ERROR] = 0
    counts = np.array([1, 0, 300, 1, 1, 0])              # slot 1 leaves: 6 pages back
    ks, vs = rows(counts)
    res = b.step(np.array([0, 1, 0, 0, 0, 0]), ks, vs, counts,
                 wl.queries(w, device="cuda", step=2))
    _check_step(b, res, 2)
    assert not res[2].any()


def test_step_latent_draft_tokens():
    """Latent layout, 4 causal draft tokens per request (each decoding slot
    appends 4 rows a step), with a stale request and joins."""
    rng = np.random.default_rng(5)
    S, T = 5, 4
    w = wl.Workload("step_lat", 44, np.zeros(S, np.int32), 16, 1, 576, 512, 64, T, 1, 200,
                    float(np.float32(1 / np.sqrt(576))), steps=1000)
    b = Both(w, 0)
    rows = _Rows(b)
    active = set()
    for rnd in range(4):
        counts = np.zeros(S, np.int64)
        for r in active:
            counts[r] = T
        free = [r for r in range(S) if r not in active]
        join = rng.choice(free, size=min(2, len(free)), replace=False)
        counts[join] = rng.integers(T, 700, len(join))
        victims = []
        if rnd == 2:
            r = sorted(active)[0]
            j = int((b.sl_h[r] - 1) // 64)
            b.et_h[r, j] = np.uint32(b.et_h[r, j]) + np.uint32(7)
            b.et_d.copy_(torch.from_numpy(b.et_h.view(np.int32)))
            victims.append(r)
        ks, vs = rows(counts)
        res = b.step(None, ks, vs, counts, wl.queries(w, device="cuda", step=rnd))
        _check_step(b, res, rnd)
        assert set(np.flatnonzero(res[2]).tolist()) == set(victims)
        active |= set(int(x) for x in join)
        active -= set(victims)


@pytest.mark.parametrize("dtype,Hq", [(0, 16), (0, 48), (1, 48)])
def test_step_in_a_cuda_graph(dtype, Hq):
    """The step launches nothing that needs the host: one captured decode
    step (one new row per slot) replayed on new rows and queries matches the
    oracle every time, including a replay in which a request goes stale and
    is removed inside the graph.  4 or 12 query rows per kv head (the 8-row
    and the 16-row consumer kernels)."""
    S = 8
    lens = np.array([37, 300, 16, 1, 700, 129, 64, 5], np.int32)
    w = wl.Workload("step_graph", 55 + Hq + dtype, lens, Hq, 4, 128, 128, 16, 1, 0, 200,
                    float(np.float32(1 / np.sqrt(128))), steps=64)
    b = Both(w, dtype)
    assert b.fill()[0] == 0
    kv = b.kv
    k_s = torch.zeros((S, 4, 128), dtype=torch.bfloat16, device="cuda")
    v_s = torch.zeros_like(k_s)
    q_s = torch.zeros((S, 1, Hq, 128), dtype=torch.bfloat16, device="cuda")
    ind = torch.arange(S + 1, dtype=torch.int32, device="cuda")
    out = torch.full((S, 1, Hq, 128), SENTINEL, dtype=torch.bfloat16, device="cuda")
    m_d = torch.zeros(S, dtype=torch.uint8, device="cuda")
    ws = torch.empty(b.dev.step_workspace_size(S, Hq, 1), dtype=torch.uint8, device="cuda")

    def launch():
        b.dev.step(S, Hq, 1, None, k_s, v_s, ind, 1, b.pt_d, b.et_d, b.sl_d, q_s, w.sm_scale, out,
                   m_d, kv.KV_STEP_REMOVE_ABORTED, ws)

    # one eager attention (it changes no pool state) does the kernels'
    # one-time attribute setup outside the capture
    b.attn(wl.queries(w, device="cuda"), None, None)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        launch()
    for rnd in range(4):
        k, v = wl.step_rows(w, rnd, device="cuda")
        q = wl.queries(w, device="cuda", step=rnd)
        k_s.copy_(k)
        v_s.copy_(v)
        q_s.copy_(q)
        out.fill_(SENTINEL)
        if rnd == 2:  # slot 4's partly filled page goes stale
            j = int((b.sl_h[4]) // 16)
            b.et_h[4, j] = np.uint32(b.et_h[4, j]) - np.uint32(1)
            b.et_d.copy_(torch.from_numpy(b.et_h.view(np.int32)))
        g.replay()

        st, m_h, ref, written = oracle.step(
            b.ref, None, wl.bits_u16(k), wl.bits_u16(v), np.arange(S + 1, dtype=np.int32), 1,
            b.pt_h, b.et_h, b.sl_h, wl.bits_u16(q), w.sm_scale, Hq, 1)
        _check_step(b, (st, m_d, m_h, out, ref, written), rnd)
        if rnd == 2:
            assert m_h.tolist() == [0, 0, 0, 0, 1, 0, 0, 0] and b.sl_h[4] == 0


@pytest.mark.parametrize("dtype,scale_mode,Hq", [(0, 0, 16), (1, 0, 16), (0, 1, 16), (0, 0, 80),
                                                 (1, 0, 80)])
def test_step_random_rounds(dtype, scale_mode, Hq):
    """Thirty random steps on a small pool: leaves, joins with prompts of up
    to a few pages, decode rows, injected stale tags, and steps that run out
    of pages (the longest request then leaves to make room).  Pool state,
    abort mask and outputs match the oracle's step after every step.  4 or
    20 query rows per kv head."""
    rng = np.random.default_rng(100 + 10 * dtype + scale_mode + Hq)
    S = 10
    w = wl.Workload("step_rand", 301 + dtype + 7 * scale_mode + Hq, np.zeros(S, np.int32), Hq, 4,
                    128, 128, 16, 1, 0, 40, float(np.float32(1 / np.sqrt(128))), steps=400,
                    magnitude=1.0)
    b = Both(w, dtype, scale_mode=scale_mode)
    rows = _Rows(b)
    mp = b.pt_h.shape[1]
    seen = {"oop": 0, "stale": 0}
    for rnd in range(30):
        live = [r for r in range(S) if b.sl_h[r] > 0]
        leave = np.zeros(S, np.uint8)
        for r in live:
            if rng.random() < 0.15:
                leave[r] = 1
        counts = np.zeros(S, np.int64)
        for r in range(S):
            if b.sl_h[r] > 0 and not leave[r]:
                counts[r] = 1
            elif rng.random() < 0.4:
                counts[r] = int(rng.integers(1, 200))
        counts = np.minimum(counts, mp * 16 - np.where(leave == 1, 0, b.sl_h))
        stale = []
        cand = [r for r in live if not leave[r]]
        if cand and rng.random() < 0.3:
            r = int(rng.choice(cand))
            j = int(rng.integers(0, -(-int(b.sl_h[r]) // 16)))
            b.et_h[r, j] = np.uint32(b.et_h[r, j]) - np.uint32(1)
            b.et_d.copy_(torch.from_numpy(b.et_h.view(np.int32)))
            stale.append(r)
            seen["stale"] += 1
        ks, vs = rows(counts)
        res = b.step(leave if leave.any() else None, ks, vs, counts,
                     wl.queries(w, device="cuda", step=rnd))
        st = res[0]
        _check_step(b, res, rnd, expect_status=st)
        assert st in (0, b.kv.KV_ERR_OUT_OF_PAGES)
        assert set(np.flatnonzero(res[2] & 1).tolist()) == set(stale)
        if st != 0:
            seen["oop"] += 1
            b.dev.ctl[b.kv.KV_CTL_ERROR] = 0
            r = int(np.argmax(b.sl_h))
            mask = np.zeros(S, np.uint8)
            mask[r] = 1
            assert b.release(mask) == 0
            torch.cuda.synchronize()
            assert b.dev.error() == 0
            b.assert_state_equal()
    assert seen["oop"] > 0 and seen["stale"] > 0, seen
