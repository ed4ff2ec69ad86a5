"""GPU parity of KV_SCALE_REQUANTIZE: a partly filled e4m3 block whose new
rows need a larger scale takes amax/448 of those rows and re-encodes its
codes.  Streams of single-token (and few-token) appends with growing
magnitude force re-quantisation again and again; cache bytes and scales must
match the oracle bit for bit, and attention over the result stays within
the usual tolerance.  A bulk append that starts in a partly filled page
takes the register-resident path and is checked the same way."""
import numpy as np
import pytest
import torch

import workloads as wl
from pathrun import Both, bf16_to_f64, close

pytestmark = pytest.mark.gpu


def _grow(w, b, steps, rows_per_step, tag0, factor=1.35):
    for st in range(steps):
        ks, vs = [], []
        for r in range(w.B):
            k, v = wl.kv_rows(w, r, 200000 + int(b.sl_h[r]), rows_per_step, device="cuda",
                              tag=tag0 + st)
            g = factor ** st
            ks.append((k.float() * g).to(torch.bfloat16))
            vs.append(None if v is None else (v.float() * g).to(torch.bfloat16))
        assert b.append(ks, vs, np.full(w.B, rows_per_step, np.int64)) == (0, w.B)
    torch.cuda.synchronize()
    assert b.dev.error() == 0


def _attn_ok(b, mag):
    """Attention within the usual bound after dividing both sides by `mag`,
    the largest factor the stream's rows were drawn at: the outputs average V
    rows of that magnitude, so the bound's absolute term scales with it (as
    in the magnitude tests)."""
    out, ref, written = b.attn(wl.queries(b.w, device="cuda"), None, None)
    got = bf16_to_f64(out.cpu().view(torch.int16).numpy().view(np.uint16))
    for r in range(b.w.B):
        if written[r]:
            ok, mabs, mrel, _ = close(got[r] / mag, ref[r] / mag)
            assert ok, f"request {r}: max abs {mabs:.3g} max rel {mrel:.3g} (relative to {mag:.3g})"


@pytest.mark.parametrize("rows_per_step", [1, 3])
def test_gqa_requantise_stream(rows_per_step):
    lens = np.array([5, 37, 16, 100, 1], np.int32)
    w = wl.Workload("requant", 71, lens, 16, 4, 128, 128, 16, 1, 0, 256,
                    float(np.float32(1 / np.sqrt(128))), steps=64)
    b = Both(w, 0, scale_mode=1)
    assert b.fill()[0] == 0
    _grow(w, b, 12, rows_per_step, 50)
    b.assert_state_equal()
    _attn_ok(b, 1.35 ** 11)


def test_latent_requantise_stream():
    lens = np.array([70, 130, 64, 3], np.int32)
    w = wl.Workload("requant_latent", 72, lens, 16, 1, 576, 512, 64, 4, 1, 64,
                    float(np.float32(1 / np.sqrt(576))), steps=64)
    b = Both(w, 0, scale_mode=1)
    assert b.fill()[0] == 0
    _grow(w, b, 10, 4, 60)
    b.assert_state_equal()
    _attn_ok(b, 1.35 ** 9)


def test_bulk_append_into_a_partial_page_requantises():
    """Requests already hold a partial page; then 100 rows each at 3x the
    magnitude (a bulk append: the first page of each request is partial)."""
    lens = np.array([5, 9, 1, 15], np.int32)
    w = wl.Workload("requant_bulk", 73, lens, 16, 8, 128, 128, 16, 1, 0, 128,
                    float(np.float32(1 / np.sqrt(128))), steps=200)
    b = Both(w, 0, scale_mode=1)
    assert b.fill()[0] == 0
    ks, vs = [], []
    for r in range(w.B):
        k, v = wl.kv_rows(w, r, int(b.sl_h[r]), 100, device="cuda", tag=9)
        ks.append((k.float() * 3).to(torch.bfloat16))
        vs.append((v.float() * 3).to(torch.bfloat16))
    assert b.append(ks, vs, np.full(w.B, 100, np.int64)) == (0, w.B)
    torch.cuda.synchronize()
    assert b.dev.error() == 0
    b.assert_state_equal()
    _attn_ok(b, 3.0)
