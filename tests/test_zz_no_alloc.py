"""paged_decode_attn_noalloc: decode attention for callers that cannot
allocate device memory (a runtime that owns all of the GPU's memory and hands
out no scratch).  Its scratch is a fixed array inside the library; the test
checks that two calls in a row, through the C ABI, give the output of the
regular entry point (which takes a caller workspace) within the attention
tolerance, and that an oversized batch is refused before any work.

Named so pytest collects it last: if it fails, a run that stops at the first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from pathrun import Both, bf16_to_f64, close

pytestmark = pytest.mark.gpu


def _bits(t):
    return bf16_to_f64(t.cpu().view(torch.int16).numpy().view(np.uint16))


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("Hq", [32, 96])
def test_noalloc_matches_workspace_entry_point_twice(dtype, Hq):
    """8 or 24 query rows per kv head (the 8-row and the 16-row kernels)."""
    lens = np.array([37, 64, 100, 255, 1, 4097, 16, 900], np.int32)
    w = wl.Workload("noalloc", 4242 + dtype + Hq, lens, Hq, 4, 128, 128, 16, 1, 0, 1024,
                    float(np.float32(1 / np.sqrt(128))), stale=[2])
    b = Both(w, dtype)
    assert b.fill()[0] == 0
    b.make_stale()
    m_d, _ = b.verify()
    q = wl.queries(w, device="cuda")
    kv = b.kv
    ref = torch.full((w.B, 1, w.num_q_heads, w.head_dim_v), 7.0, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(b.dev.workspace_size(w.B, w.num_q_heads, 1), dtype=torch.uint8, device="cuda")
    kv.paged_decode_attn(b.dev.handle, w.B, w.num_q_heads, 1, q, b.pt_d, b.sl_d, m_d, w.sm_scale,
                         ref, ws)
    want = _bits(ref)
    for _ in range(2):
        out = torch.full_like(ref, 7.0)
        kv.paged_decode_attn_noalloc(b.dev.handle, w.B, w.num_q_heads, 1, q, b.pt_d, b.sl_d, m_d,
                                     w.sm_scale, out)
        got = _bits(out)
        for r in range(w.B):
            if m_d[r].item():
                assert np.all(got[r] == 7.0)  # aborted: untouched, as with the workspace call
            else:
                ok, mabs, mrel, _ = close(got[r], want[r])
                assert ok, (r, mabs, mrel)
    assert b.dev.error() == 0


def test_noalloc_latent_layout():
    """The same for the latent (tensor-core) path: 4 draft tokens x 16 heads on
    one 576-wide row per token."""
    lens = np.array([37, 300, 64, 1000], np.int32)
    w = wl.Workload("noalloc_lat", 4343, lens, 16, 1, 576, 512, 64, 4, 1, 64,
                    float(np.float32(1 / np.sqrt(576))))
    b = Both(w, 0)
    assert b.fill()[0] == 0
    q = wl.queries(w, device="cuda")
    kv = b.kv
    shape = (w.B, 4, 16, 512)
    ref = torch.full(shape, 7.0, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(b.dev.workspace_size(w.B, 16, 4), dtype=torch.uint8, device="cuda")
    kv.paged_decode_attn(b.dev.handle, w.B, 16, 4, q, b.pt_d, b.sl_d, None, w.sm_scale, ref, ws)
    want = _bits(ref)
    out = torch.full(shape, 7.0, dtype=torch.bfloat16, device="cuda")
    kv.paged_decode_attn_noalloc(b.dev.handle, w.B, 16, 4, q, b.pt_d, b.sl_d, None, w.sm_scale,
                                 out)
    got = _bits(out)
    for r in range(w.B):
        ok, mabs, mrel, _ = close(got[r], want[r])
        assert ok, (r, mabs, mrel)
    assert b.dev.error() == 0


def test_noalloc_refuses_batches_beyond_its_scratch():
    import paged_fp8_kv_append_gb300 as kv

    pool = kv.KVPool(64, 16, 8, 128, 128, device="cuda")
    B = 8192  # needs far more than the fixed scratch
    assert pool.workspace_size(B, 64, 1) > 32 << 20
    with pytest.raises(kv.KVError) as e:
        kv.paged_decode_attn_noalloc(
            pool.handle, B, 64, 1, torch.zeros((B, 1, 64, 128), dtype=torch.bfloat16, device="cuda"),
            torch.zeros((B, 4), dtype=torch.int32, device="cuda"),
            torch.zeros(B, dtype=torch.int32, device="cuda"), None, 0.1,
            torch.zeros((B, 1, 64, 128), dtype=torch.bfloat16, device="cuda"))
    assert e.value.status == kv.KV_ERR_UNSUPPORTED
    assert pool.error() == 0  # nothing was enqueued
