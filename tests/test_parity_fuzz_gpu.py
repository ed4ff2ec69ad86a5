"""Randomised parity of the whole GQA path against the oracle: seeded draws
of batch size, lengths (empty and partly filled pages included), draft
tokens, query-group sizes up to 64 rows per kv head, an injected stale tag,
e4m3 and bf16 pools.  Every draw: append (bulk or decode-size), tag check,
attention; pool state bit-exact, attention within the tolerance, aborted and
empty requests as specified ("Smaller, faster, safer: running Kimi and GLM at
scale", sections "Quantizing the KV cache" and "Protecting a shared KV
cache")."""
import numpy as np
import pytest
import torch

import workloads as wl
from pathrun import Both, bf16_to_f64, close

pytestmark = pytest.mark.gpu


def _draw(rng):
    Hkv = int(rng.choice([1, 2, 4, 8]))
    while True:
        G = int(rng.integers(1, 17))
        T = int(rng.integers(1, 5))
        if T * G <= 64:
            break
    B = int(rng.integers(1, 10))
    lens = rng.integers(0, 700, B).astype(np.int32)
    lens[rng.random(B) < 0.15] = 0
    lens = np.where((lens > 0) & (lens < T), T, lens).astype(np.int32)
    return B, Hkv, G, T, lens


@pytest.mark.parametrize("seed", range(12))
def test_random_shapes(seed):
    rng = np.random.default_rng(9000 + seed)
    B, Hkv, G, T, lens = _draw(rng)
    dtype = seed % 2
    npg = int((-(-lens.astype(np.int64) // 16)).sum()) + 16
    w = wl.Workload("fuzz", 7000 + seed, lens, Hkv * G, Hkv, 128, 128, 16, T, 0, npg,
                    float(np.float32(1 / np.sqrt(128))), steps=8)
    b = Both(w, dtype)
    assert b.fill()[0] == 0
    live = [r for r in range(B) if lens[r] > 0]
    stale = []
    if live and rng.random() < 0.5:
        r = int(rng.choice(live))
        j = int(rng.integers(0, -(-int(lens[r]) // 16)))
        b.et_h[r, j] = np.uint32(b.et_h[r, j]) - np.uint32(1)
        b.et_d.copy_(torch.from_numpy(b.et_h.view(np.int32)))
        stale.append(r)
    torch.cuda.synchronize()
    b.assert_state_equal()
    m_d, m_h = b.verify()
    assert np.array_equal(m_d.cpu().numpy(), m_h)
    assert set(np.flatnonzero(m_h).tolist()) == set(stale)
    out, ref, written = b.attn(wl.queries(w, device="cuda"), m_d, m_h)
    assert b.dev.error() == 0
    got = bf16_to_f64(out.cpu().view(torch.int16).numpy().view(np.uint16))
    for r in range(B):
        if m_h[r]:
            assert np.all(got[r] == 7.0)
        else:
            assert written[r]
            ok, mabs, mrel, _ = close(got[r], ref[r])
            assert ok, (seed, r, mabs, mrel, (B, Hkv, G, T, dtype))
