"""GPU parity for bf16 queries outside f16's comfortable range.  The e4m3
kernels multiply in f16 (every e4m3 code is exact in f16); the bf16 query
("Smaller, faster, safer: running Kimi and GLM at scale", section
"Quantizing the KV cache": the cache is FP8, the query stays BF16) is scaled
per row by an exact power of two before it is narrowed, so rows at 1e6
(beyond f16's 65504) and at 1e-6 (f16 subnormals) still match the fp64
oracle within |o - r| <= 2e-3 + 1e-2 |r|.  Also one row with a single large
element among ordinary ones."""
import dataclasses

import numpy as np
import pytest
import torch

import workloads as wl
from pathrun import Both, bf16_to_f64, close

pytestmark = pytest.mark.gpu


def _check(b, q):
    w = b.w
    out, ref, written = b.attn(q, None, None)
    got = bf16_to_f64(out.cpu().view(torch.int16).numpy().view(np.uint16))
    assert np.isfinite(got).all()
    for r in range(w.B):
        assert written[r]
        ok, mabs, mrel, _ = close(got[r], ref[r])
        assert ok, (r, mabs, mrel)
    assert b.dev.error() == 0


@pytest.mark.parametrize("mag", [1e6, 1e-6, "spike"])
@pytest.mark.parametrize("Hq", [8, 24])
def test_gqa_e4m3_query_range(mag, Hq):
    """8 query rows per kv head (8-row kernel) and 12 (16-row kernel)."""
    w = dataclasses.replace(wl.tiny(seed=4601 + Hq), num_q_heads=Hq)
    b = Both(w, 0)
    assert b.fill()[0] == 0
    q = wl.queries(w, device="cuda").float()
    if mag == "spike":
        q[:, :, 0, 5] = 3.0e4  # one large element in one row of every request
        q[:, :, 1, :] *= 1e5   # and a whole row beyond f16's range
    else:
        q *= mag
    _check(b, q.to(torch.bfloat16))


@pytest.mark.parametrize("mag", [1e6, 1e-6])
def test_latent_query_range(mag):
    lens = np.array([37, 300, 64, 1000], np.int32)
    w = wl.Workload("qrange_lat", 4707, lens, 16, 1, 576, 512, 64, 4, 1, 64,
                    float(np.float32(1 / np.sqrt(576))))
    b = Both(w, 0)
    assert b.fill()[0] == 0
    q = (wl.queries(w, device="cuda").float() * mag).to(torch.bfloat16)
    _check(b, q)
