"""GPU parity of the latent (MLA-style) path: 576-wide e4m3 rows per token
(the first 512 dims are V), one scale per page, T causal draft tokens per
request, tcgen05 tensor cores.  Cache bytes and scales bit-exact; outputs
within |o - r| <= 2e-3 + 1e-2 |r| of the fp64 oracle."""
import os

import numpy as np
import pytest
import torch

import workloads as wl
from pathrun import Both, FullSize, bf16_to_f64, close

pytestmark = pytest.mark.gpu


def _lat(lens, T, Hq, seed=3, magnitude=1.0):
    lens = np.array(lens, np.int32)
    npg = int((-(-lens.astype(np.int64) // 64)).sum()) + 8
    return wl.Workload("latent", seed, lens, Hq, 1, 576, 512, 64, T, 1, npg,
                       float(np.float32(1 / np.sqrt(576))), magnitude=magnitude)


def _check(out, ref, written, sentinel=7.0):
    got = bf16_to_f64(out.cpu().view(torch.int16).numpy().view(np.uint16))
    for r in range(len(written)):
        if written[r]:
            ok, mabs, mrel, _ = close(got[r], ref[r])
            assert ok, f"request {r}: max abs {mabs:.3g} max rel {mrel:.3g}"
        else:
            assert np.all(got[r] == sentinel)


@pytest.mark.parametrize("T,Hq,lens", [
    (4, 16, [37, 300, 64, 65, 1, 4]),        # one 64-row block per request
    (1, 64, [129, 33, 500]),                 # plain decode, one block
    (2, 64, [1000, 2, 77]),                  # two blocks per request
    (4, 128, [90, 700]),                     # eight blocks (the verify shape)
])
def test_latent_small(T, Hq, lens):
    w = _lat(lens, T, Hq, seed=7 + T + Hq)
    b = Both(w, 0)
    assert b.fill()[0] == 0
    torch.cuda.synchronize()
    b.assert_state_equal()
    out, ref, written = b.attn(wl.queries(w, device="cuda"), None, None)
    assert b.dev.error() == 0, b.kv.kv_status_string(b.dev.error())
    _check(out, ref, written)


@pytest.mark.parametrize("mag", [1e-4, 3e3])
def test_latent_magnitude_extremes(mag):
    """Cache rows drawn at 1e-4 and 3e3 (page scales about 1e-6 and 30): the
    attention weights must stay in f16's normal range.  Compared relative to
    the magnitude."""
    w = _lat([300, 1000, 65, 7], 4, 16, seed=21, magnitude=mag)
    b = Both(w, 0)
    assert b.fill()[0] == 0
    torch.cuda.synchronize()
    b.assert_state_equal()
    out, ref, written = b.attn(wl.queries(w, device="cuda"), None, None)
    assert written.all() and b.dev.error() == 0
    got = bf16_to_f64(out.cpu().view(torch.int16).numpy().view(np.uint16))
    for r in range(w.B):
        ok, mabs, mrel, _ = close(got[r] / mag, ref[r] / mag)
        assert ok, f"request {r}: max abs {mabs:.3g} max rel {mrel:.3g} (relative to {mag})"


def test_latent_ring_wraps_and_abort():
    """Many units per CTA (the rings wrap many times); an aborted request is
    skipped and left untouched; a bad page id in a request is not read."""
    w = _lat([20000, 15000, 900, 6000], 4, 16, seed=11)
    b = Both(w, 0)
    assert b.fill()[0] == 0
    q = wl.queries(w, device="cuda")
    mask_h = np.array([0, 1, 0, 0], np.uint8)
    mask_d = torch.from_numpy(mask_h).cuda()
    out, ref, written = b.attn(q, mask_d, mask_h)
    assert written.tolist() == [1, 0, 1, 1]
    assert b.dev.error() == 0
    _check(out, ref, written)
    b.pt_h[2, 3] = 10 ** 8
    b.pt_d[2, 3] = 10 ** 8
    out, ref, written = b.attn(q, None, None)
    assert written.tolist() == [1, 1, 0, 1]
    _check(out, ref, written)
    assert b.dev.error() == b.kv.KV_ERR_BAD_PAGE_ID


def test_latent_verify_full_size_sampled():
    """The 64-request latent verify workload (lognormal contexts 8k..64k, 128
    heads x 4 draft tokens) at full size; the oracle checks a seeded subset
    of 8 requests, every head and draft token, cache codes and scales bit
    for bit."""
    w = wl.latent_verify()
    kvp = __import__("paged_fp8_kv_append_gb300")
    dev = kvp.KVPool(w.num_pages, 64, 1, 576, 512, dtype=0, layout=1, device="cuda",
                     tags=wl.initial_tags(w), free_list=wl.free_list(w))
    B, mp = w.B, w.max_pages
    pt = torch.full((B, mp), -1, dtype=torch.int32, device="cuda")
    et = torch.zeros((B, mp), dtype=torch.int32, device="cuda")
    sl = torch.zeros(B, dtype=torch.int32, device="cuda")
    for r0 in range(0, B, 8):
        counts = np.zeros(B, np.int64)
        ks = []
        for r in range(r0, min(B, r0 + 8)):
            counts[r] = int(w.lens[r])
            ks.append(wl.kv_rows(w, r, 0, int(counts[r]), device="cuda")[0])
        ind = torch.from_numpy(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)).cuda()
        dev.append(B, torch.cat(ks), None, ind, int(counts.max()), pt, et, sl)
    q = wl.queries(w, device="cuda")
    out = torch.zeros((B, 4, 128, 512), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(dev.workspace_size(B, 128, 4), dtype=torch.uint8, device="cuda")
    dev.attn(B, 128, 4, q, pt, sl, None, w.sm_scale, out, ws)
    torch.cuda.synchronize()
    assert dev.error() == 0

    # a seeded subset of 8 requests, every head and draft token, the oracle
    # runs in a process pool (spawn: the parent has touched the GPU)
    import multiprocessing as mp

    from pathrun import latent_oracle_request

    rng = np.random.default_rng(2)
    chosen = sorted(rng.choice(B, 8, replace=False).tolist())
    got_all = bf16_to_f64(out.cpu().view(torch.int16).numpy().view(np.uint16))
    jobs = []
    for r in chosen:
        L = int(w.lens[r])
        rows = wl.bits_u16(wl.kv_rows(w, r, 0, L, device="cuda")[0])
        jobs.append((rows, L, wl.bits_u16(q[r:r + 1]), w.sm_scale, 128, 4))
    with mp.get_context("spawn").Pool(min(8, os.cpu_count() or 1)) as pool_:
        results = pool_.map(latent_oracle_request, jobs)
    for r, (codes, scales, ref) in zip(chosen, results):
        L = int(w.lens[r])
        pages = torch.from_numpy(pt[r, : -(-L // 64)].cpu().numpy().astype(np.int64)).cuda()
        assert np.array_equal(dev.k_cache[pages].cpu().numpy(), codes), r
        assert np.array_equal(dev.k_scale[pages].cpu().numpy().view(np.uint32), scales.view(np.uint32)), r
        ok, mabs, mrel, _ = close(got_all[r], ref)
        assert ok, (r, mabs, mrel)
