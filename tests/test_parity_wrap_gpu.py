"""GPU parity with many units of work per CTA, so the split kernel's
shared-memory ring wraps several times and requests span several CTAs, for
every head-group size (8, 4, 2, 1 kv heads per unit) and both cache dtypes;
and the same with more than 8 query rows per kv head (warps of 16 rows,
one or two per kv head)."""
import numpy as np
import pytest
import torch

import workloads as wl
from pathrun import Both, bf16_to_f64, close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("Hkv,Hq", [(8, 16), (4, 16), (2, 4), (6, 12), (16, 16)])
def test_ring_wraps(dtype, Hkv, Hq):
    lens = np.array([9000, 7003, 20000, 3001, 1], np.int32)
    w = wl.Workload("wrap", 515 + Hkv, lens, Hq, Hkv, 128, 128, 16, 1, 0,
                    int(lens.sum() // 16 + 64), float(np.float32(1 / np.sqrt(128))))
    b = Both(w, dtype)
    assert b.fill()[0] == 0
    out, ref, written = b.attn(wl.queries(w, device="cuda"), None, None)
    assert b.dev.error() == 0, b.kv.kv_status_string(b.dev.error())
    got = bf16_to_f64(out.cpu().view(torch.int16).numpy().view(np.uint16))
    for r in range(w.B):
        ok, mabs, mrel, _ = close(got[r], ref[r])
        assert ok, (r, mabs, mrel)


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("T,Hq,Hkv", [(1, 96, 8), (4, 64, 8), (2, 16, 1), (3, 36, 4),
                                      (4, 64, 4)])
def test_ring_wraps_wide_groups(dtype, T, Hq, Hkv):
    R = T * Hq // Hkv
    lens = np.array([9000, 7003, 20000, 3001, 1, 5000], np.int32)
    w = wl.Workload("wrapwide", 733 + R, lens, Hq, Hkv, 128, 128, 16, T, 0,
                    int(lens.sum() // 16 + 64), float(np.float32(1 / np.sqrt(128))))
    b = Both(w, dtype)
    assert b.fill()[0] == 0
    out, ref, written = b.attn(wl.queries(w, device="cuda"), None, None)
    assert b.dev.error() == 0, b.kv.kv_status_string(b.dev.error())
    got = bf16_to_f64(out.cpu().view(torch.int16).numpy().view(np.uint16))
    for r in range(w.B):
        ok, mabs, mrel, _ = close(got[r], ref[r])
        assert ok, (r, mabs, mrel)
