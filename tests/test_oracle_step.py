"""Oracle pins for the continuous-batching step ("Smaller, faster, safer:
running Kimi and GLM at scale", section "Protecting a shared KV cache": the
tag check is on for every step while requests come and go, and a request
whose pages were reallocated is aborted and returns no data).

The bookkeeping below is worked out by hand from the rules the oracle states
(pops from free_list[free_head], tag += 1 per pop, release pushes pages back
below free_head in (request, page) order).  The values are pinned against
the separately pinned append and attention on a batch built without the
aborted request's rows, which is what the step must reduce to."""
import numpy as np
import torch

import oracle

P = 4


def bf16_bits(x):
    t = torch.tensor(np.asarray(x, np.float64), dtype=torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _ind(ns):
    return np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)


def _pool(n=8, H=1, D=16, layout=0):
    tags = [10 * (i + 1) for i in range(n)]
    fl = [5, 2, 7, 0, 3, 6, 1, 4] + list(range(8, n))
    if layout == 0:
        return oracle.Pool(n, P, H, D, D, dtype=0, layout=0, tags=tags, free_list=fl)
    return oracle.Pool(n, P, 1, D, D // 2, dtype=0, layout=1, tags=tags, free_list=fl)


def _rows(rng, n, H=1, D=16):
    return bf16_bits(rng.standard_normal((n, H, D))), bf16_bits(rng.standard_normal((n, H, D)))


def _k_rows(pool, pt_row, n):
    """K codes of a request's first n tokens: [n][H][D] (K pages are [H][P][D])."""
    return np.stack([pool.k_cache[pt_row[i // P], :, i % P, :] for i in range(n)])


def _v_rows(pool, pt_row, n):
    """V codes of a request's first n tokens: [n][H][D] (V pages are [H][D][P])."""
    return np.stack([pool.v_cache[pt_row[i // P], :, :, i % P] for i in range(n)])


def test_step_by_hand():
    """Slot 0 leaves and a new request joins it, slot 1 went stale, slot 2
    was empty and a request joins it."""
    rng = np.random.default_rng(1)
    pool = _pool()
    B, mp = 3, 4
    pt, et, sl = np.full((B, mp), -1, np.int32), np.zeros((B, mp), np.uint32), np.zeros(B, np.int32)
    k, v = _rows(rng, 8)
    assert oracle.append(pool, k, v, _ind([5, 3, 0]), 5, pt, et, sl) == (0, 3)
    assert pt[:, :2].tolist() == [[5, 2], [7, -1], [-1, -1]] and int(pool.free_head[0]) == 3
    pool.tags[7] += 1  # slot 1's page was handed out elsewhere
    page7 = (pool.k_cache[7].copy(), pool.v_cache[7].copy())

    k, v = _rows(rng, 2 + 1 + 6)
    q = bf16_bits(rng.standard_normal((B, 1, 2, 16)))
    st, mask, out, written = oracle.step(
        pool, np.array([1, 0, 0], np.uint8), k, v, _ind([2, 1, 6]), 6, pt, et, sl, q,
        0.25, 2, 1)
    assert st == 0                       # the stale slot is dropped, not an append error
    assert mask.tolist() == [0, oracle.ABORT_TAG, 0]
    assert written.tolist() == [1, 0, 1]
    # slot 0 released pages 5, 2 (head 3 -> 1); slot 0 pops 5 (tag 62),
    # slot 2 pops 2 (tag 32) and 0 (tag 11); slot 1 is released at the end
    assert pt.tolist() == [[5, -1, -1, -1], [-1] * 4, [2, 0, -1, -1]]
    assert et.tolist() == [[62, 0, 0, 0], [0] * 4, [32, 11, 0, 0]]
    assert sl.tolist() == [2, 0, 6]
    assert int(pool.free_head[0]) == 3 and pool.free_list[3] == 7
    assert pool.tags.tolist() == [11, 20, 32, 40, 50, 62, 70, 82]
    assert np.array_equal(pool.k_cache[7], page7[0]) and np.array_equal(pool.v_cache[7], page7[1])
    # the joined slots hold exactly what a fresh pool makes of the same rows
    for r, rows in ((0, slice(0, 2)), (2, slice(3, 9))):
        fresh = oracle.Pool(4, P, 1, 16, 16, dtype=0, layout=0)
        n = rows.stop - rows.start
        fpt, fet, fsl = np.full((1, 4), -1, np.int32), np.zeros((1, 4), np.uint32), np.zeros(1, np.int32)
        assert oracle.append(fresh, k[rows], v[rows], _ind([n]), n, fpt, fet, fsl) == (0, 1)
        npg = -(-n // P)
        # the written rows (a reused page keeps its old bytes past them)
        assert np.array_equal(_k_rows(pool, pt[r], n), _k_rows(fresh, fpt[0], n))
        assert np.array_equal(_v_rows(pool, pt[r], n), _v_rows(fresh, fpt[0], n))
        assert np.array_equal(pool.k_scale[pt[r, :npg]], fresh.k_scale[fpt[0, :npg]])
        assert np.array_equal(pool.v_scale[pt[r, :npg]], fresh.v_scale[fpt[0, :npg]])


def test_step_reduces_to_append_and_attention_without_the_stale_request():
    """Everything the step does for the other requests equals a plain append
    in which the stale request has no rows, followed by attention with that
    request masked."""
    rng = np.random.default_rng(2)
    B, mp, H, G = 5, 8, 2, 2
    lens = [9, 6, 13, 3, 0]
    k0, v0 = _rows(rng, sum(lens), H)
    new = [1, 1, 1, 5, 7]
    k1, v1 = _rows(rng, sum(new), H)
    q = bf16_bits(rng.standard_normal((B, 1, H * G, 16)))
    runs = []
    for mode in ("step", "plain"):
        pool = _pool(40, H)
        pt, et, sl = np.full((B, mp), -1, np.int32), np.zeros((B, mp), np.uint32), np.zeros(B, np.int32)
        assert oracle.append(pool, k0, v0, _ind(lens), 13, pt, et, sl) == (0, B)
        pool.tags[pt[2, 1]] += 1         # request 2: an inner page went stale
        pool.tags[pt[1, 1]] += 1         # request 1: its partly filled page went stale
        if mode == "step":
            st, mask, out, written = oracle.step(pool, None, k1, v1, _ind(new), 7, pt, et, sl,
                                                 q, 0.3, H * G, 1, remove_aborted=False)
            assert st == 0 and mask.tolist() == [0, 1, 1, 0, 0]
        else:
            ind = np.array(_ind(new), np.int64)
            keep = [0, 3, 4]
            kk = np.concatenate([k1[ind[r]:ind[r + 1]] for r in keep])
            vv = np.concatenate([v1[ind[r]:ind[r + 1]] for r in keep])
            cnt = [new[r] if r in keep else 0 for r in range(B)]
            assert oracle.append(pool, kk, vv, _ind(cnt), 7, pt, et, sl) == (0, B)
            out, written = oracle.attn(pool, q, pt, sl, np.array([0, 1, 1, 0, 0], np.uint8), 0.3,
                                       H * G, 1)
        runs.append((pool, pt, et, sl, out, written))
    (a, *ra), (b, *rb) = runs
    for x, y in zip(ra, rb):
        assert np.array_equal(x, y)
    for f in ("k_cache", "v_cache", "k_scale", "v_scale", "tags", "free_list", "free_head"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f


def test_step_out_of_pages_marks_the_rest_unserved():
    """The append stops at the first request the free list cannot serve;
    that request and every later one are marked unserved, attend nothing,
    keep their state, and are not released."""
    rng = np.random.default_rng(3)
    pool = _pool(8)
    B, mp = 4, 6
    pt, et, sl = np.full((B, mp), -1, np.int32), np.zeros((B, mp), np.uint32), np.zeros(B, np.int32)
    k, v = _rows(rng, 4 + 4 + 1 + 1)
    assert oracle.append(pool, k, v, _ind([4, 4, 1, 1]), 4, pt, et, sl) == (0, B)
    assert int(pool.free_head[0]) == 4
    snap = (pt.copy(), et.copy(), sl.copy())
    # request 0 needs 1 page, request 1 needs 4 (only 3 are left)
    k, v = _rows(rng, 1 + 13 + 1 + 1)
    q = bf16_bits(rng.standard_normal((B, 1, 1, 16)))
    st, mask, out, written = oracle.step(pool, None, k, v, _ind([1, 13, 1, 1]), 13, pt, et, sl,
                                         q, 0.25, 1, 1)
    assert st == oracle.ERR_OUT_OF_PAGES
    assert mask.tolist() == [0, 2, 2, 2] and written.tolist() == [1, 0, 0, 0]
    assert sl.tolist() == [5, 4, 1, 1] and int(pool.free_head[0]) == 5
    assert np.array_equal(pt[1:], snap[0][1:]) and np.array_equal(et[1:], snap[1][1:])


def test_step_latent_two_draft_tokens():
    """Latent layout (one row per token, V = its first dims): the step is
    append then attention when no request leaves or aborts."""
    rng = np.random.default_rng(4)
    B, mp, T = 3, 6, 2
    lens = [7, 0, 12]
    k0 = bf16_bits(rng.standard_normal((sum(lens), 16)))
    new = [T, T, T]
    k1 = bf16_bits(rng.standard_normal((sum(new), 16)))
    q = bf16_bits(rng.standard_normal((B, T, 4, 16)))
    res = []
    for mode in ("step", "plain"):
        pool = _pool(20, layout=1)
        pt, et, sl = np.full((B, mp), -1, np.int32), np.zeros((B, mp), np.uint32), np.zeros(B, np.int32)
        assert oracle.append(pool, k0, None, _ind(lens), 12, pt, et, sl) == (0, B)
        if mode == "step":
            st, mask, out, written = oracle.step(pool, None, k1, None, _ind(new), T, pt, et, sl,
                                                 q, 0.2, 4, T)
            assert st == 0 and not mask.any()
        else:
            assert oracle.append(pool, k1, None, _ind(new), T, pt, et, sl) == (0, B)
            out, written = oracle.attn(pool, q, pt, sl, None, 0.2, 4, T)
        res.append((pool.k_cache.copy(), pool.k_scale.copy(), pt, sl, out, written))
    for x, y in zip(*res):
        assert np.array_equal(x, y)
    assert res[0][5].tolist() == [1, 1, 1]


def _check_invariants(pool, pt, et, sl):
    """Page conservation and consistency after a step: the free list's tail
    and the live mappings together hold every page exactly once, every live
    mapping carries its page's current tag, and each request maps exactly
    its first ceil(L / P) entries."""
    head = int(pool.free_head[0])
    free = pool.free_list[head:].tolist()
    mapped = []
    for r in range(len(sl)):
        n = -(-int(sl[r]) // P)
        assert all(p >= 0 for p in pt[r, :n]) and all(p == -1 for p in pt[r, n:]), r
        mapped += pt[r, :n].tolist()
        for j in range(n):
            assert et[r, j] == pool.tags[pt[r, j]], (r, j)
    assert sorted(free + mapped) == list(range(pool.num_pages))


def test_step_random_sequence_invariants():
    """Forty random steps (leaves, joins, decode rows, injected stale tags,
    runs out of pages now and then): after every step the pool is
    consistent, the aborted set is exactly the injected stale requests and
    the unserved ones are exactly those at or after the append's stop."""
    rng = np.random.default_rng(7)
    B, mp = 6, 12
    pool = _pool(24)
    pt, et, sl = np.full((B, mp), -1, np.int32), np.zeros((B, mp), np.uint32), np.zeros(B, np.int32)
    saw = {"oop": 0, "stale": 0, "join": 0}
    for step in range(40):
        live = [r for r in range(B) if sl[r] > 0]
        leave = np.zeros(B, np.uint8)
        for r in live:
            if rng.random() < 0.15:
                leave[r] = 1
        counts = np.zeros(B, np.int64)
        for r in range(B):
            if sl[r] > 0 and not leave[r]:
                counts[r] = 1
            elif rng.random() < 0.5:
                counts[r] = int(rng.integers(1, 30))  # a new request's prompt
                saw["join"] += 1
        counts = np.minimum(counts, mp * P - np.where(leave == 1, 0, sl))
        stale = []
        cand = [r for r in live if not leave[r]]
        if cand and rng.random() < 0.3:
            r = int(rng.choice(cand))
            j = int(rng.integers(0, -(-int(sl[r]) // P)))
            et[r, j] -= np.uint32(1)
            stale.append(r)
            saw["stale"] += 1
        k, v = _rows(rng, int(counts.sum()) or 1)
        q = bf16_bits(rng.standard_normal((B, 1, 1, 16)))
        st, mask, out, written = oracle.step(pool, leave if leave.any() else None, k, v,
                                             _ind(counts), int(max(counts.max(), 1)), pt, et, sl,
                                             q, 0.25, 1, 1)
        assert st in (oracle.OK, oracle.ERR_OUT_OF_PAGES)
        assert set(np.flatnonzero(mask & oracle.ABORT_TAG).tolist()) == set(stale)
        unserved = np.flatnonzero(mask & oracle.ABORT_UNSERVED).tolist()
        if st == oracle.ERR_OUT_OF_PAGES:
            saw["oop"] += 1
            assert unserved and unserved == list(range(unserved[0], B))
        else:
            assert not unserved
        assert [r for r in range(B) if written[r]] == [r for r in range(B) if mask[r] == 0]
        for r in stale:
            assert sl[r] == 0  # removed in the same step
        _check_invariants(pool, pt, et, sl)
        if st == oracle.ERR_OUT_OF_PAGES:  # make room: the longest request leaves
            r = int(np.argmax(sl))
            assert oracle.release(pool, pt, et, sl, np.eye(B, dtype=np.uint8)[r]) == 0
            _check_invariants(pool, pt, et, sl)
    assert saw["oop"] > 0 and saw["stale"] > 0 and saw["join"] > 0, saw
