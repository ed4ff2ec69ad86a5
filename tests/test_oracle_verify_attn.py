"""Pins for the oracle's tag check and fp64 decode attention.

Tag check: section "Protecting a shared KV cache" of "Smaller, faster, safer:
running Kimi and GLM at scale" -- every page has a tag that changes on
reallocation; each request's expected (page, tag) list is checked before the
decode reads the cache; a mismatch aborts exactly that request.  Pinned by a
brute-force restatement in Python on small random cases and by invariants.

Attention: section "Quantizing the KV cache" -- the attention reads the e4m3
cache and converts values as it reads them.  Pinned against
torch.nn.functional.scaled_dot_product_attention in float64 (a library routine)
on K/V gathered and dequantised with torch's float8 decode, plus closed-form
special cases (one token returns V, constant V returns the constant, page
permutation and head-group invariance, the textbook causal mask).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def bf16_bits(x):
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).to(torch.float64)


# -------------------------------------------------------------------- verify

def _verify_brute(num_pages, P, tags, pt, et, sl):
    out = []
    for r in range(len(sl)):
        L = int(sl[r])
        if L < 0 or -(-L // P) > pt.shape[1]:
            out.append(1)
            continue
        bad = 0
        for j in range(-(-L // P)):
            p = int(pt[r, j])
            if not (0 <= p < num_pages) or int(tags[p]) != int(et[r, j]):
                bad = 1
        out.append(bad)
    return np.array(out, np.uint8)


@pytest.mark.parametrize("seed", range(6))
def test_verify_brute_force_random(seed):
    rng = np.random.default_rng(seed)
    npg, P, B, mp = 40, 4, 9, 6
    tags = rng.integers(0, 2 ** 32, npg, dtype=np.uint64).astype(np.uint32)
    pt = rng.integers(0, npg, (B, mp)).astype(np.int32)
    et = tags[pt].copy()
    sl = rng.integers(0, mp * P + 1, B).astype(np.int32)
    # corruptions: stale tags, out-of-range ids, entries past the length (ignored)
    for _ in range(4):
        r, j = rng.integers(B), rng.integers(mp)
        kind = rng.integers(3)
        if kind == 0:
            et[r, j] -= np.uint32(1)
        elif kind == 1:
            pt[r, j] = rng.choice([-1, npg, npg + 7])
        else:
            et[r, j] ^= np.uint32(1 << int(rng.integers(32)))
    sl[0] = -1
    got = oracle.verify(npg, P, tags, pt, et, sl)
    assert np.array_equal(got, _verify_brute(npg, P, tags, pt, et, sl))
    assert got[0] == 1


def test_verify_invariants():
    rng = np.random.default_rng(11)
    npg, P, B, mp = 64, 16, 4, 16
    tags = rng.integers(0, 2 ** 32, npg, dtype=np.uint64).astype(np.uint32)
    perm = rng.permutation(npg).astype(np.int32)
    pt = perm[: B * mp].reshape(B, mp).copy()
    et = tags[pt].copy()
    sl = np.array([37, 64, 100, 255], np.int32)
    assert oracle.verify(npg, P, tags, pt, et, sl).tolist() == [0, 0, 0, 0]
    # one stale tag in request 2 aborts exactly request 2
    et2 = et.copy()
    et2[2, 3] = tags[pt[2, 3]] - np.uint32(1)
    assert oracle.verify(npg, P, tags, pt, et2, sl).tolist() == [0, 0, 1, 0]
    # a stale entry beyond the request's pages is not checked
    et3 = et.copy()
    et3[0, 5] ^= np.uint32(1)  # request 0 uses pages 0..2 only
    assert oracle.verify(npg, P, tags, pt, et3, sl).tolist() == [0, 0, 0, 0]
    # an out-of-range id aborts, without reading past the tag array
    pt4 = pt.copy()
    pt4[1, 0] = npg + 1000
    assert oracle.verify(npg, P, tags, pt4, et, sl).tolist() == [0, 1, 0, 0]
    # reallocating a page (tag += 1) aborts every request that still maps it
    tags5 = tags.copy()
    tags5[pt[3, 7]] += np.uint32(1)
    assert oracle.verify(npg, P, tags5, pt, et, sl).tolist() == [0, 0, 0, 1]


# ----------------------------------------------------------------- attention

def _build(rng, dtype, lens, Hkv=2, G=4, D=32, P=4, T=1, free=None, scale_std=None):
    """Fill an oracle pool through oracle.append and return everything."""
    B = len(lens)
    npg = sum(-(-L // P) for L in lens) + 3
    pool = oracle.Pool(npg, P, Hkv, D, D, dtype=dtype,
                       free_list=free if free is not None else rng.permutation(npg))
    ind = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    std = scale_std if scale_std is not None else np.ones((1, Hkv, D))
    k = bf16_bits(rng.standard_normal((ind[-1], Hkv, D)) * std)
    v = bf16_bits(rng.standard_normal((ind[-1], Hkv, D)) * std)
    mp = max(-(-L // P) for L in lens) + 1
    pt = np.full((B, mp), -1, np.int32)
    et = np.zeros((B, mp), np.uint32)
    sl = np.zeros(B, np.int32)
    st, stop = oracle.append(pool, k, v, ind, max(max(lens), 1), pt, et, sl)
    assert st == 0 and stop == B
    q = bf16_bits(rng.standard_normal((B, T, Hkv * G, D)))
    return pool, pt, sl, q


def _gather_deq(pool, pt, r, L):
    """[Hkv][L][D] K and V, dequantised with torch (library decode)."""
    P = pool.page_size
    pages = pt[r, : -(-L // P)]
    if pool.dtype == 0:
        kc = torch.from_numpy(pool.k_cache[pages]).view(torch.float8_e4m3fn).to(torch.float32)
        vc = torch.from_numpy(pool.v_cache[pages]).view(torch.float8_e4m3fn).to(torch.float32)
        ks = torch.from_numpy(pool.k_scale[pages])[:, :, None, None]
        vs = torch.from_numpy(pool.v_scale[pages])[:, :, None, None]
        k = (kc * ks).to(torch.float64)            # fp32 product, then widened
        v = (vc * vs).to(torch.float64)
    else:
        k = bits_to_f64(pool.k_cache[pages])
        v = bits_to_f64(pool.v_cache[pages])
    # k: [pages][H][P][D] -> [H][pages*P][D]; v: [pages][H][D][P] -> [H][pages*P][D]
    k = k.permute(1, 0, 2, 3).reshape(pool.num_kv_heads, -1, pool.dk)[:, :L]
    v = v.permute(1, 0, 3, 2).reshape(pool.num_kv_heads, -1, pool.dv)[:, :L]
    return k, v


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("T", [1, 3])
def test_attn_vs_sdpa_float64(dtype, T):
    rng = np.random.default_rng(100 + dtype * 10 + T)
    lens = [1, 5, 13, 40, 3]
    Hkv, G, D = 2, 4, 32
    pool, pt, sl, q = _build(rng, dtype, lens, Hkv=Hkv, G=G, D=D, T=T,
                             scale_std=rng.uniform(0.5, 4, (1, Hkv, D)))
    sm = np.float32(1.0 / math.sqrt(D))
    out, wr = oracle.attn(pool, q, pt, sl, None, sm, Hkv * G, T)
    assert wr.tolist() == [1] * len(lens)
    for r, L in enumerate(lens):
        k, v = _gather_deq(pool, pt, r, L)
        k = k.repeat_interleave(G, dim=0)  # query head h reads kv head h // G
        v = v.repeat_interleave(G, dim=0)
        qh = bits_to_f64(q[r]).permute(1, 0, 2)  # [Hq][T][D]
        # query token i sees positions 0 .. L - T + i
        pos = torch.arange(L)
        allowed = pos[None, :] <= (L - T + torch.arange(T))[:, None]
        ref = torch.zeros(Hkv * G, T, D, dtype=torch.float64)
        rows = allowed.any(dim=1)
        if rows.any():
            ref[:, rows] = F.scaled_dot_product_attention(
                qh[:, rows], k, v, attn_mask=allowed[rows], scale=float(sm))
        got = torch.from_numpy(out[r]).permute(1, 0, 2)
        assert torch.allclose(got, ref, rtol=1e-12, atol=1e-12), (r, (got - ref).abs().max())


def test_single_token_returns_v_and_constant_v():
    rng = np.random.default_rng(5)
    pool, pt, sl, q = _build(rng, 0, [1, 9], Hkv=1, G=2, D=16)
    out, _ = oracle.attn(pool, q, pt, sl, None, 0.25, 2, 1)
    k, v = _gather_deq(pool, pt, 0, 1)
    assert np.array_equal(out[0, 0, 0], v[0, 0].numpy()) and np.array_equal(out[0, 0, 1], v[0, 0].numpy())
    # constant V (bf16 cache, all rows equal) returns that constant
    P = 4
    pool2 = oracle.Pool(8, P, 1, 16, 16, dtype=1)
    L = 11
    vrow = bf16_bits(rng.standard_normal(16))
    kk = bf16_bits(rng.standard_normal((L, 1, 16)) * 3)
    vv = np.broadcast_to(vrow, (L, 1, 16)).copy()
    pt2 = np.full((1, 4), -1, np.int32)
    sl2 = np.zeros(1, np.int32)
    oracle.append(pool2, kk, vv, np.array([0, L]), L, pt2, np.zeros((1, 4), np.uint32), sl2)
    q2 = bf16_bits(rng.standard_normal((1, 1, 3, 16)))
    out2, _ = oracle.attn(pool2, q2, pt2, sl2, None, 0.5, 3, 1)
    c = bits_to_f64(vrow).numpy()
    assert np.allclose(out2[0, 0], c[None, :], rtol=0, atol=1e-15)


def test_page_permutation_and_group_invariance():
    rng = np.random.default_rng(9)
    lens = [23, 7]
    npg = sum(-(-L // 4) for L in lens) + 3
    free_a = np.arange(npg)
    free_b = np.random.default_rng(1).permutation(npg)
    pool_a, pt_a, sl, q = _build(np.random.default_rng(2), 0, lens, free=free_a)
    pool_b, pt_b, _, _ = _build(np.random.default_rng(2), 0, lens, free=free_b)
    # identical logical content in different physical pages: identical output
    oa, _ = oracle.attn(pool_a, q, pt_a, sl, None, 0.2, 8, 1)
    ob, _ = oracle.attn(pool_b, q, pt_b, sl, None, 0.2, 8, 1)
    assert np.array_equal(oa, ob)
    # identical q in two heads of one group: identical output rows
    q2 = q.copy()
    q2[:, :, 1] = q2[:, :, 0]
    o2, _ = oracle.attn(pool_a, q2, pt_a, sl, None, 0.2, 8, 1)
    assert np.array_equal(o2[:, :, 0], o2[:, :, 1])


def test_causal_T4_L4_is_textbook_causal():
    rng = np.random.default_rng(4)
    pool, pt, sl, q = _build(rng, 1, [4], Hkv=1, G=3, D=8, P=2, T=4)
    out, _ = oracle.attn(pool, q, pt, sl, None, 0.3, 3, 4)
    k, v = _gather_deq(pool, pt, 0, 4)
    qh = bits_to_f64(q[0]).permute(1, 0, 2)
    ref = F.scaled_dot_product_attention(qh, k.expand(3, -1, -1), v.expand(3, -1, -1),
                                         is_causal=True, scale=float(np.float32(0.3)))
    assert torch.allclose(torch.from_numpy(out[0]).permute(1, 0, 2), ref, rtol=1e-12, atol=1e-13)


def test_abort_and_empty_and_bad_page():
    rng = np.random.default_rng(8)
    pool, pt, sl, q = _build(rng, 0, [6, 6, 6], Hkv=1, G=2, D=16, T=2)
    out, wr = oracle.attn(pool, q, pt, sl, np.array([0, 1, 0], np.uint8), 0.3, 2, 2)
    assert wr.tolist() == [1, 0, 1] and np.all(out[1] == 0)
    # fewer positions than query tokens: query 0 sees nothing -> zero row
    sl1 = sl.copy()
    sl1[0] = 1
    out1, _ = oracle.attn(pool, q, pt, sl1, None, 0.3, 2, 2)
    assert np.all(out1[0, 0] == 0) and np.any(out1[0, 1] != 0)
    # a bad page id in a request the check did not abort: no output either
    pt2 = pt.copy()
    pt2[2, 1] = 10_000
    _, wr2 = oracle.attn(pool, q, pt2, sl, None, 0.3, 2, 2)
    assert wr2.tolist() == [1, 1, 0]


def test_latent_vs_sdpa():
    rng = np.random.default_rng(21)
    P, Dk, Dv, Hq, T = 8, 40, 32, 6, 4
    lens = [4, 19, 33]
    npg = sum(-(-L // P) for L in lens) + 2
    pool = oracle.Pool(npg, P, 1, Dk, Dv, dtype=0, layout=1, free_list=rng.permutation(npg))
    ind = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    kv = bf16_bits(rng.standard_normal((ind[-1], Dk)))
    pt = np.full((3, 6), -1, np.int32)
    sl = np.zeros(3, np.int32)
    oracle.append(pool, kv, None, ind, 40, pt, np.zeros((3, 6), np.uint32), sl)
    q = bf16_bits(rng.standard_normal((3, T, Hq, Dk)))
    sm = np.float32(1 / math.sqrt(Dk))
    out, wr = oracle.attn(pool, q, pt, sl, None, sm, Hq, T)
    for r, L in enumerate(lens):
        pages = pt[r, : -(-L // P)]
        c = torch.from_numpy(pool.k_cache[pages]).view(torch.float8_e4m3fn).to(torch.float32)
        c = (c * torch.from_numpy(pool.k_scale[pages])[:, None, None]).to(torch.float64)
        rows = c.reshape(-1, Dk)[:L]
        qh = bits_to_f64(q[r]).permute(1, 0, 2)
        allowed = torch.arange(L)[None, :] <= (L - T + torch.arange(T))[:, None]
        ref = F.scaled_dot_product_attention(qh, rows.expand(Hq, -1, -1),
                                             rows[:, :Dv].expand(Hq, -1, -1),
                                             attn_mask=allowed, scale=float(sm))
        assert torch.allclose(torch.from_numpy(out[r]).permute(1, 0, 2), ref, rtol=1e-12, atol=1e-12)
