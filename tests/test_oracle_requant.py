"""Oracle pins for scale_mode 1 (re-quantise a partly filled block when new
rows need a larger scale) against mode 0 (frozen scale, later rows saturate).

The pages only say the cache is held as FP8 e4m3 ("Smaller, faster, safer:
running Kimi and GLM at scale", section "Quantizing the KV cache"); both
modes are this library's readings.  Every value below is exact in bf16 and
every scale is exact in fp32 (amax 112 -> 0.25, 224 -> 0.5, 336 -> 0.75,
1.75 -> 2^-8), so each code is read off the OFP8 E4M3 table by hand:
0x7E = 448, 0x76 = 224, 0x72 = 160, 0x71 = 144, 0x70 = 128, 0x54 = 12,
0x4C = 6."""
import numpy as np
import torch

import oracle

P, D = 4, 16


def _bits(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def _rows(first_vals, n):
    """n rows [row][1 head][D]; row i gets first_vals[i] in dim 0, else zeros
    except a 3.0 in dim 1 of row 0."""
    x = np.zeros((n, 1, D), np.float32)
    for i, v in enumerate(first_vals):
        x[i, 0, 0] = v
    return x


def _append(pool, k, v, pt, et, sl, n):
    ind = np.array([0, n], np.int32)
    return oracle.append(pool, _bits(k), _bits(v), ind, n, pt, et, sl)


def _setup(mode):
    pool = oracle.Pool(4, P, 1, D, D, dtype=0, layout=0, scale_mode=mode)
    pt, et, sl = np.full((1, 4), -1, np.int32), np.zeros((1, 4), np.uint32), np.zeros(1, np.int32)
    k = _rows([112.0, 0.0], 2)
    k[0, 0, 1] = 3.0
    v = _rows([1.75, 0.0], 2)
    assert _append(pool, k, v, pt, et, sl, 2) == (0, 1)
    p = int(pt[0, 0])
    assert pool.k_scale[p, 0] == 0.25 and pool.v_scale[p, 0] == 2.0 ** -8
    assert pool.k_cache[p, 0, 0, :2].tolist() == [0x7E, 0x54]
    assert pool.v_cache[p, 0, 0, 0] == 0x7E
    return pool, pt, et, sl, p


def test_requantise_when_a_row_needs_a_larger_scale():
    pool, pt, et, sl, p = _setup(1)
    k, v = _rows([224.0], 1), _rows([0.5], 1)
    assert _append(pool, k, v, pt, et, sl, 1) == (0, 1)
    # K: scale 0.25 -> 0.5; 448*0.25 = 112 -> 224 (0x76), 12*0.25 = 3 -> 6 (0x4C)
    assert pool.k_scale[p, 0] == 0.5
    assert pool.k_cache[p, 0, 0, :2].tolist() == [0x76, 0x4C]
    assert pool.k_cache[p, 0, 2, 0] == 0x7E           # the new row: 224 / 0.5 = 448
    # V: 0.5 needs scale 0.5/448 < 2^-8, so the scale and old codes stay
    assert pool.v_scale[p, 0] == 2.0 ** -8
    assert pool.v_cache[p, 0, 0, 0] == 0x7E and pool.v_cache[p, 0, 0, 2] == 0x70  # 0.5*256 = 128


def test_frozen_scale_saturates_instead():
    pool, pt, et, sl, p = _setup(0)
    assert _append(pool, _rows([224.0], 1), _rows([0.5], 1), pt, et, sl, 1) == (0, 1)
    assert pool.k_scale[p, 0] == 0.25
    assert pool.k_cache[p, 0, 0, :2].tolist() == [0x7E, 0x54]
    assert pool.k_cache[p, 0, 2, 0] == 0x7E           # 224 / 0.25 = 896 saturates to 448


def test_requantise_rounds_again():
    """Ratio 3: 448 * 0.25 = 112, 112 / 0.75 = 149.33 -> nearest code 144 (0x71)."""
    pool, pt, et, sl, p = _setup(1)
    assert _append(pool, _rows([336.0], 1), _rows([0.0], 1), pt, et, sl, 1) == (0, 1)
    assert pool.k_scale[p, 0] == 0.75
    assert pool.k_cache[p, 0, 0, 0] == 0x71 and pool.k_cache[p, 0, 2, 0] == 0x7E
    # 3.0 * ... : 12 * 0.25 = 3 -> 3 / 0.75 = 4 (0x48: E=9, M=0 -> 4)
    assert pool.k_cache[p, 0, 0, 1] == 0x48


def test_requantise_latent_page():
    pool = oracle.Pool(4, P, 1, D, D, dtype=0, layout=1, scale_mode=1)
    pt, et, sl = np.full((1, 4), -1, np.int32), np.zeros((1, 4), np.uint32), np.zeros(1, np.int32)
    x = np.zeros((2, D), np.float32)
    x[0, 0], x[1, 5] = 112.0, 3.0
    ind = np.array([0, 2], np.int32)
    assert oracle.append(pool, _bits(x), None, ind, 2, pt, et, sl) == (0, 1)
    p = int(pt[0, 0])
    assert pool.k_scale[p] == 0.25 and pool.k_cache[p, 0, 0] == 0x7E and pool.k_cache[p, 1, 5] == 0x54
    y = np.zeros((1, D), np.float32)
    y[0, 3] = 224.0
    assert oracle.append(pool, _bits(y), None, np.array([0, 1], np.int32), 1, pt, et, sl) == (0, 1)
    assert pool.k_scale[p] == 0.5
    assert pool.k_cache[p, 0, 0] == 0x76 and pool.k_cache[p, 1, 5] == 0x4C
    assert pool.k_cache[p, 2, 3] == 0x7E
