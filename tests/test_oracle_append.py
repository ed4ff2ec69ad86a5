"""Pins for the oracle's append: page allocation, tag stamping (section
"Protecting a shared KV cache" of "Smaller, faster, safer: running Kimi and GLM
at scale": a page's tag changes whenever it is reallocated) and quantise-on-write
into the FP8 e4m3 cache (section "Quantizing the KV cache").

The expected values of the tiny cases are enumerated by hand from the e4m3
definition; the random cases check invariants computed with torch (amax,
float8 decode) rather than with the oracle's own code.
"""
import numpy as np
import pytest
import torch

import oracle


def bf16_bits(x):
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f32(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).float().numpy()


def fp8_to_f64(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _tiny_pool(**kw):
    return oracle.Pool(num_pages=4, page_size=2, num_kv_heads=1, dk=2, dv=2,
                       tags=[10, 20, 30, 40], free_list=[2, 0, 3, 1], **kw)


def test_tiny_hand_enumerated_append():
    pool = _tiny_pool()
    B, max_pages = 2, 3
    pt = np.full((B, max_pages), -1, np.int32)
    et = np.zeros((B, max_pages), np.uint32)
    sl = np.zeros(B, np.int32)
    # request 0: 3 rows, request 1: 1 row
    k = bf16_bits([[[1.0, -2.0]], [[0.5, 4.0]], [[3.0, 0.0]], [[-1.0, 1.0]]])
    v = bf16_bits([[[2.0, 2.0]], [[-1.0, 0.0]], [[0.0, 0.0]], [[7.0, -7.0]]])
    st, stop = oracle.append(pool, k, v, np.array([0, 3, 4]), 3, pt, et, sl)
    assert (st, stop) == (0, 2)
    # pops in request order: r0 <- pages 2, 0 ; r1 <- page 3 ; tag += 1 each
    assert pt.tolist() == [[2, 0, -1], [3, -1, -1]]
    assert et.tolist() == [[31, 11, 0], [41, 0, 0]]
    assert pool.tags.tolist() == [11, 20, 31, 41]
    assert int(pool.free_head[0]) == 3 and sl.tolist() == [3, 1]
    # page 2, K: amax 4 -> scale 4/448; 1/s=112 -> 0x6E, -2/s=-224 -> 0xF6,
    # 0.5/s=56 -> 0x66, 4/s=448 -> 0x7E
    assert pool.k_scale[2, 0] == np.float32(4.0) / np.float32(448.0)
    assert pool.k_cache[2, 0].tolist() == [[0x6E, 0xF6], [0x66, 0x7E]]
    # page 2, V (dim-major): amax 2 -> 2/s = 448 -> 0x7E ; -1/s=-224 -> 0xF6 ; 0 -> 0x00
    assert pool.v_cache[2, 0].tolist() == [[0x7E, 0xF6], [0x7E, 0x00]]
    # page 0 holds r0's third row: K amax 3 -> 3/s = 448 -> 0x7E, 0 -> 0x00;
    # V is all zero -> amax 0 -> scale 1.0, codes 0
    assert pool.k_scale[0, 0] == np.float32(3.0) / np.float32(448.0)
    assert pool.k_cache[0, 0, 0].tolist() == [0x7E, 0x00]
    assert pool.v_scale[0, 0] == 1.0 and pool.v_cache[0, 0, :, 0].tolist() == [0, 0]
    # page 3 (r1): K [-1, 1] -> [0xFE, 0x7E]; V [7, -7] -> [0x7E, 0xFE]
    assert pool.k_cache[3, 0, 0].tolist() == [0xFE, 0x7E]
    assert pool.v_cache[3, 0, :, 0].tolist() == [0x7E, 0xFE]

    # second call: r0 appends [8, 0.25] into its partly filled page 0 whose
    # K scale stays 3/448: 8/s saturates (0x7E); 0.25/s = 37.33 -> 1.125*2^5 = 0x61
    k2 = bf16_bits([[[8.0, 0.25]]])
    v2 = bf16_bits([[[0.0, 0.0]]])
    st, stop = oracle.append(pool, k2, v2, np.array([0, 1, 1]), 1, pt, et, sl)
    assert (st, stop) == (0, 2)
    assert pool.k_scale[0, 0] == np.float32(3.0) / np.float32(448.0)
    assert pool.k_cache[0, 0, 1].tolist() == [0x7E, 0x61]
    assert pool.tags.tolist() == [11, 20, 31, 41] and int(pool.free_head[0]) == 3
    assert sl.tolist() == [4, 1]


def test_out_of_pages_stops_at_that_request():
    pool = _tiny_pool()
    B, max_pages = 3, 4
    pt = np.full((B, max_pages), -1, np.int32)
    et = np.zeros((B, max_pages), np.uint32)
    sl = np.zeros(B, np.int32)
    rows = [2, 7, 1]  # needs 1 + 4 + 1 pages; only 4 exist
    ind = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    k = bf16_bits(np.ones((ind[-1], 1, 2)))
    st, stop = oracle.append(pool, k, k, ind, 8, pt, et, sl)
    assert st == oracle.ERR_OUT_OF_PAGES and stop == 1
    assert sl.tolist() == [2, 0, 0] and int(pool.free_head[0]) == 1
    assert pool.tags.tolist() == [10, 20, 31, 40]
    assert pt[1:].tolist() == [[-1] * 4, [-1] * 4]


def test_bad_free_list_entry_and_invalid_args_stop():
    pool = oracle.Pool(num_pages=4, page_size=2, num_kv_heads=1, dk=2, dv=2,
                       free_list=[1, 9, 0, 2])
    pt = np.full((2, 4), -1, np.int32)
    et = np.zeros((2, 4), np.uint32)
    sl = np.zeros(2, np.int32)
    k = bf16_bits(np.ones((4, 1, 2)))
    st, stop = oracle.append(pool, k, k, np.array([0, 2, 4]), 4, pt, et, sl)
    assert st == oracle.ERR_BAD_PAGE_ID and stop == 1 and sl.tolist() == [2, 0]
    # request longer than max_pages * P
    pool2 = _tiny_pool()
    pt2 = np.full((1, 1), -1, np.int32)
    st, stop = oracle.append(pool2, k, k, np.array([0, 3]), 4, pt2, np.zeros((1, 1), np.uint32),
                             np.zeros(1, np.int32))
    assert st == oracle.ERR_INVALID_ARG and stop == 0
    # more rows than max_new
    st, stop = oracle.append(_tiny_pool(), k, k, np.array([0, 3]), 2, np.full((1, 4), -1, np.int32),
                             np.zeros((1, 4), np.uint32), np.zeros(1, np.int32))
    assert st == oracle.ERR_INVALID_ARG and stop == 0


def test_tag_wraps_mod_2_32():
    pool = oracle.Pool(num_pages=2, page_size=4, num_kv_heads=1, dk=2, dv=2,
                       tags=[0xFFFFFFFF, 5], free_list=[0, 1])
    pt = np.full((1, 2), -1, np.int32)
    et = np.zeros((1, 2), np.uint32)
    k = bf16_bits(np.ones((1, 1, 2)))
    oracle.append(pool, k, k, np.array([0, 1]), 1, pt, et, np.zeros(1, np.int32))
    assert pool.tags[0] == 0 and et[0, 0] == 0


@pytest.mark.parametrize("dtype", [0, 1])
def test_random_gather_back_invariants(dtype):
    """Gathering each request's rows back through its page table gives the
    per-(page, head) quantisation of the inputs (e4m3) or the inputs (bf16)."""
    rng = np.random.default_rng(7)
    P, H, D, npg = 4, 2, 16, 64
    pool = oracle.Pool(npg, P, H, D, D, dtype=dtype, free_list=rng.permutation(npg))
    lens = [5, 12, 1, 0, 9]
    B = len(lens)
    ind = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    kf = (rng.standard_normal((ind[-1], H, D)) * rng.uniform(0.5, 4, (1, H, D))).astype(np.float32)
    vf = rng.standard_normal((ind[-1], H, D)).astype(np.float32)
    k, v = bf16_bits(kf), bf16_bits(vf)
    pt = np.full((B, 8), -1, np.int32)
    et = np.zeros((B, 8), np.uint32)
    sl = np.zeros(B, np.int32)
    st, stop = oracle.append(pool, k, v, ind, 16, pt, et, sl)
    assert st == 0 and stop == B and sl.tolist() == lens
    kx, vx = bits_to_f32(k), bits_to_f32(v)
    for r in range(B):
        for pos in range(lens[r]):
            p, slot = pt[r, pos // P], pos % P
            row = ind[r] + pos
            for h in range(H):
                kcode = pool.k_cache[p, h, slot]
                vcode = pool.v_cache[p, h, :, slot]
                if dtype == 1:
                    assert np.array_equal(kcode, k[row, h]) and np.array_equal(vcode, v[row, h])
                    continue
                # scale == fl32(torch amax over the page's rows / 448)
                rows = slice(ind[r] + (pos // P) * P, ind[r] + min(lens[r], (pos // P + 1) * P))
                kam = torch.from_numpy(kx[rows, h]).abs().max().item()
                assert pool.k_scale[p, h] == np.float32(kam) / np.float32(448.0)
                deq = fp8_to_f64(kcode) * float(pool.k_scale[p, h])
                err = np.abs(deq - kx[row, h])
                assert np.all(err <= 2.0 ** -4 * np.abs(kx[row, h]) + float(pool.k_scale[p, h]) * 2.0 ** -10 + 1e-12)
                deqv = fp8_to_f64(vcode) * float(pool.v_scale[p, h])
                assert np.all(np.abs(deqv - vx[row, h]) <= 2.0 ** -4 * np.abs(vx[row, h])
                              + float(pool.v_scale[p, h]) * 2.0 ** -10 + 1e-12)
    # every popped page has tag == expected tag
    for r in range(B):
        for j in range(-(-lens[r] // P)):
            assert pool.tags[pt[r, j]] == et[r, j]


def test_latent_scale_per_page_over_all_dims():
    rng = np.random.default_rng(3)
    P, Dk = 4, 24
    pool = oracle.Pool(8, P, 1, Dk, 16, dtype=0, layout=1)
    x = rng.standard_normal((6, Dk)).astype(np.float32)
    x[2, 20] = 9.0  # amax in a dim beyond dv: it still sets the page scale
    kb = bf16_bits(x)
    pt = np.full((1, 4), -1, np.int32)
    st, _ = oracle.append(pool, kb, None, np.array([0, 6]), 6, pt, np.zeros((1, 4), np.uint32),
                          np.zeros(1, np.int32))
    assert st == 0
    assert pool.k_scale[pt[0, 0]] == np.float32(9.0) / np.float32(448.0)
    assert pool.k_cache[pt[0, 0], 2, 20] == 0x7E
    xf = bits_to_f32(kb)
    am2 = np.abs(xf[4:6]).max()
    assert pool.k_scale[pt[0, 1]] == np.float32(am2) / np.float32(448.0)


def test_fp8_pool_holds_twice_the_tokens():
    """Section "Quantizing the KV cache": e4m3 halves the cache size.  Bytes per
    token for Hkv=8, D=128, P=16: 2048 (+ 8 scales per page = 4 B/token)
    against 4096 for bf16, i.e. capacity ratio 4096/2052 ~ 1.996."""
    fp8 = oracle.Pool(16, 16, 8, 128, 128, dtype=0)
    bf = oracle.Pool(16, 16, 8, 128, 128, dtype=1)
    tok = 16 * 16
    b8 = (fp8.k_cache.nbytes + fp8.v_cache.nbytes + fp8.k_scale.nbytes + fp8.v_scale.nbytes) / tok
    b16 = (bf.k_cache.nbytes + bf.v_cache.nbytes) / tok
    assert b8 == 2052 and b16 == 4096
    assert abs(b16 / b8 - 1.996) < 1e-3


def test_append_refuses_a_length_past_int32():
    """seq_lens are int32: an append that would take a request past 2^31 - 1
    tokens is refused (INVALID_ARG) even when the declared page-table width
    could hold it, and nothing changes.  (A page-aligned length and an
    exhausted free list, so no entry of the small page table is touched
    whichever check fires.)"""
    import ctypes

    lib = oracle._load()
    P, mp = 16, 2 ** 27 + 1                       # mp * P > 2^31
    tags = np.zeros(8, np.uint32)
    free = np.arange(8, dtype=np.int32)
    head = np.full(1, 8, np.int32)                # every page handed out: nothing is popped
    pt = np.full(4, -1, np.int32)                 # only the declared width is large
    et = np.zeros(4, np.uint32)
    sl = np.array([2 ** 31 - 16], np.int32)       # page-aligned, one page short of 2^31
    stop = np.zeros(1, np.int32)
    ind = np.array([0, 16], np.int32)             # 16 more rows would reach 2^31
    p = oracle._p
    st = lib.or_alloc(8, P, p(tags), p(free), p(head), 1, p(ind), 16, p(pt), p(et), mp, p(sl),
                      p(stop), None)
    assert st == oracle.ERR_INVALID_ARG and int(stop[0]) == 0
    assert int(head[0]) == 8 and sl.tolist() == [2 ** 31 - 16] and not tags.any()


def test_no_write_into_a_partial_page_a_later_request_of_the_call_pops():
    """Rows are written after all of the call's pops: a partly filled page
    that a later request of the same call pops (its tag changes) is not
    written through the earlier request's now stale mapping; the new owner's
    rows and scale are its own.  Worked out by hand on a P = 2 pool."""
    pool = _tiny_pool()  # tags [10, 20, 30, 40], free list [2, 0, 3, 1]
    pt = np.full((2, 3), -1, np.int32)
    et = np.zeros((2, 3), np.uint32)
    sl = np.zeros(2, np.int32)
    k = bf16_bits([[[1.0, 2.0]], [[1.0, 1.0]], [[1.0, 1.0]]])
    assert oracle.append(pool, k, k, np.array([0, 1, 3]), 2, pt, et, sl) == (0, 2)
    # request 0: page 2 (tag 31), 1 of 2 slots; request 1: page 0 (tag 11), full
    assert pt.tolist() == [[2, -1, -1], [0, -1, -1]] and et[:, 0].tolist() == [31, 11]
    assert int(pool.free_head[0]) == 2
    pool.free_list[2] = 2  # request 0's partly filled page is listed free again
    k2 = bf16_bits([[[4.0, 0.5]], [[2.0, -1.0]]])
    st, stop = oracle.append(pool, k2, k2, np.array([0, 1, 2]), 1, pt, et, sl)
    # request 0's check at its turn sees tag 31 (served); request 1 then pops
    # page 2 (tag 32) for its new logical page 1
    assert (st, stop) == (0, 2)
    assert sl.tolist() == [2, 3] and int(pool.free_head[0]) == 3 and int(pool.tags[2]) == 32
    assert pt.tolist() == [[2, -1, -1], [0, 2, -1]]
    assert et.tolist() == [[31, 0, 0], [11, 32, 0]]
    # page 2 holds request 1's row in slot 0 with its own scale 2/448:
    # 2 / (2/448) = 448 -> 0x7E, -1 / (2/448) = -224 = -1.75 * 2^7 -> 0xF6;
    # slot 1 (request 0's row) is not written
    assert pool.k_scale[2, 0] == np.float32(2.0) / np.float32(448.0)
    assert pool.k_cache[2, 0, 0].tolist() == [0x7E, 0xF6]
    assert pool.k_cache[2, 0, 1].tolist() == [0, 0]
    assert pool.v_cache[2, 0, :, 0].tolist() == [0x7E, 0xF6]
    assert pool.v_cache[2, 0, :, 1].tolist() == [0, 0]


def test_latent_no_write_into_a_partial_page_a_later_request_pops():
    """The latent layout follows the same rule: one scale per page, set by
    the new owner's rows alone."""
    pool = oracle.Pool(num_pages=4, page_size=2, num_kv_heads=1, dk=4, dv=2, layout=1,
                       tags=[10, 20, 30, 40], free_list=[2, 0, 3, 1])
    pt = np.full((2, 3), -1, np.int32)
    et = np.zeros((2, 3), np.uint32)
    sl = np.zeros(2, np.int32)
    rows = bf16_bits([[1.0, 2.0, 0.0, 0.0], [1.0, 1.0, 1.0, 1.0], [1.0, 1.0, 1.0, 1.0]])
    assert oracle.append(pool, rows, None, np.array([0, 1, 3]), 2, pt, et, sl) == (0, 2)
    assert pt[:, 0].tolist() == [2, 0]
    pool.free_list[2] = 2  # request 0's partly filled page is listed free again
    rows2 = bf16_bits([[64.0, 0.5, 0.0, 0.0], [2.0, -1.0, 0.0, 0.25]])
    st, stop = oracle.append(pool, rows2, None, np.array([0, 1, 2]), 1, pt, et, sl)
    assert (st, stop) == (0, 2) and sl.tolist() == [2, 3]
    assert pt.tolist() == [[2, -1, -1], [0, 2, -1]] and int(pool.tags[2]) == 32
    # page 2: request 1's row in slot 0 with scale 2/448 (amax over all 4 dims):
    # [448, -224, 0, 0.25 * 224 = 56 = 1.75 * 2^5] -> [0x7E, 0xF6, 0x00, 0x66];
    # slot 1 (request 0's row, which would have needed a scale of 64/448) not written
    assert pool.k_scale[2] == np.float32(2.0) / np.float32(448.0)
    assert pool.k_cache[2, 0].tolist() == [0x7E, 0xF6, 0x00, 0x66]
    assert pool.k_cache[2, 1].tolist() == [0, 0, 0, 0]


def test_latent_bf16_pool_holds_the_rows_bits():
    """A bf16 latent pool (the prefill pool a handoff reads from) keeps every
    row's bits in the slot its position names (page = page_table[r][pos / P],
    slot = pos % P), across two calls, the second into partly filled pages;
    pages no call wrote stay zero and no scale is set."""
    rng = np.random.default_rng(17)
    P, Dk, B = 4, 8, 3
    pool = oracle.Pool(12, P, 1, Dk, 8, dtype=1, layout=1, free_list=rng.permutation(12))
    pt = np.full((B, 5), -1, np.int32)
    et = np.zeros((B, 5), np.uint32)
    sl = np.zeros(B, np.int32)
    rows = [[] for _ in range(B)]
    for counts in ([5, 0, 3], [6, 2, 1]):
        kb = rng.integers(0, 2 ** 16, (sum(counts), Dk)).astype(np.uint16)
        ind = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        for r in range(B):
            rows[r].extend(kb[ind[r]:ind[r + 1]])
        st, stop = oracle.append(pool, kb, None, ind, max(counts), pt, et, sl)
        assert (st, stop) == (0, B)
    want = np.zeros_like(pool.k_cache)
    for r in range(B):
        for pos, row in enumerate(rows[r]):
            want[pt[r, pos // P], pos % P] = row
    assert sl.tolist() == [11, 2, 4]
    assert np.array_equal(pool.k_cache, want)
    assert not pool.k_scale.any()
