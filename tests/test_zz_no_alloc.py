"""paged_decode_attn_noalloc: decode attention for callers that cannot
allocate device memory (a runtime that owns all of the GPU's memory and hands
out no scratch).  Its scratch is a fixed array inside the library that every
call shares.  The tests call it through the C ABI twice, with a call of
another shape in between (so the array holds that call's leftovers), and
check each output bit for bit against the regular entry point (which takes a
caller workspace and launches the same kernels) and against the oracle
within the attention tolerance; an oversized batch is refused before any
work.

Named so pytest collects it last: if it fails, a run that stops at the first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from pathrun import Both, bf16_to_f64, close

pytestmark = pytest.mark.gpu


def _raw(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _check(got_raw, want_raw, ref, written, sentinel=7.0):
    # same kernels, grid and plan as the workspace entry point: identical bits
    assert np.array_equal(got_raw, want_raw)
    got = bf16_to_f64(got_raw)
    for r in range(got.shape[0]):
        if written[r]:
            ok, mabs, mrel, _ = close(got[r], ref[r])
            assert ok, (r, mabs, mrel)
        else:
            assert np.all(got[r] == sentinel)  # aborted: untouched


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("Hq", [32, 96])
def test_noalloc_matches_workspace_entry_point_and_oracle(dtype, Hq):
    """8 or 24 query rows per kv head (the 8-row and the 16-row kernels)."""
    lens = np.array([37, 64, 100, 255, 1, 4097, 16, 900], np.int32)
    w = wl.Workload("noalloc", 4242 + dtype + Hq, lens, Hq, 4, 128, 128, 16, 1, 0, 1024,
                    float(np.float32(1 / np.sqrt(128))), stale=[2])
    b = Both(w, dtype)
    assert b.fill()[0] == 0
    b.make_stale()
    m_d, m_h = b.verify()
    assert np.array_equal(m_d.cpu().numpy(), m_h)
    q = wl.queries(w, device="cuda")
    kv = b.kv
    ref_out, ref, written = b.attn(q, m_d, m_h)  # workspace entry point and oracle
    want = _raw(ref_out)
    # a call of another shape between the two: a different kernel, plan and
    # partial layout, so the shared array keeps different contents
    hq_other = 64 if Hq == 32 else 16
    g = torch.Generator(device="cuda")
    g.manual_seed(99 + Hq)
    q_other = torch.randn((w.B, 1, hq_other, 128), generator=g, device="cuda").to(torch.bfloat16)
    for call in range(2):
        out = torch.full_like(ref_out, 7.0)
        kv.paged_decode_attn_noalloc(b.dev.handle, w.B, w.num_q_heads, 1, q, b.pt_d, b.sl_d, m_d,
                                     w.sm_scale, out)
        _check(_raw(out), want, ref, written)
        if call == 0:
            other = torch.zeros((w.B, 1, hq_other, 128), dtype=torch.bfloat16, device="cuda")
            kv.paged_decode_attn_noalloc(b.dev.handle, w.B, hq_other, 1, q_other, b.pt_d, b.sl_d,
                                         None, w.sm_scale, other)
    assert b.dev.error() == 0


def test_noalloc_latent_layout():
    """The same for the latent (tensor-core) path: 4 draft tokens x 16 heads on
    one 576-wide row per token; the call in between attends only the first
    two requests."""
    lens = np.array([37, 300, 64, 1000], np.int32)
    w = wl.Workload("noalloc_lat", 4343, lens, 16, 1, 576, 512, 64, 4, 1, 64,
                    float(np.float32(1 / np.sqrt(576))))
    b = Both(w, 0)
    assert b.fill()[0] == 0
    q = wl.queries(w, device="cuda")
    kv = b.kv
    ref_out, ref, written = b.attn(q, None, None)
    want = _raw(ref_out)
    for call in range(2):
        out = torch.full_like(ref_out, 7.0)
        kv.paged_decode_attn_noalloc(b.dev.handle, w.B, 16, 4, q, b.pt_d, b.sl_d, None,
                                     w.sm_scale, out)
        _check(_raw(out), want, ref, written)
        if call == 0:
            other = torch.zeros_like(ref_out[:2])
            kv.paged_decode_attn_noalloc(b.dev.handle, 2, 16, 4, q[:2].contiguous(), b.pt_d,
                                         b.sl_d, None, w.sm_scale, other)
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
