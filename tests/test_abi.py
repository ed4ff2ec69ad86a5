"""The C-ABI library loads, exports every symbol the header declares, and
rejects bad arguments synchronously (no GPU needed: nothing is enqueued)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kv():
    import __graft_entry__

    __graft_entry__.build()
    import paged_fp8_kv_append_gb300 as kv

    return kv


def _declared():
    text = open(os.path.join(ROOT, "include", "kvfp8.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_0-9]+)\s*\(", text)) - {"if", "sizeof"})


def test_exports_every_declared_symbol(kv):
    names = _declared()
    assert {"kv_pool_create", "kv_append_quantize", "kv_verify_tags", "paged_decode_attn"} <= set(names)
    lib = ctypes.CDLL(kv.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def _desc(kv, **over):
    d = kv.kv_pool_desc()
    d.num_pages, d.page_size, d.num_kv_heads, d.head_dim_k, d.head_dim_v = 64, 16, 2, 128, 128
    d.dtype, d.layout = kv.KV_DTYPE_E4M3, kv.KV_LAYOUT_GQA
    fake = 0x10000  # 16-byte aligned, never dereferenced by pool creation
    d.k_cache = d.v_cache = d.k_scale = d.v_scale = d.tags = d.free_list = d.ctl = fake
    for k, v in over.items():
        setattr(d, k, v)
    return d


def test_pool_create_validation(kv):
    h = kv.kv_pool_create(_desc(kv))
    assert h
    kv.kv_pool_destroy(h)
    for bad in [dict(num_pages=0), dict(page_size=0), dict(head_dim_k=100), dict(dtype=7),
                dict(layout=3), dict(k_cache=None), dict(v_scale=None), dict(ctl=0x10004),
                dict(layout=1, num_kv_heads=2)]:
        with pytest.raises(kv.KVError) as e:
            kv.kv_pool_create(_desc(kv, **bad))
        assert e.value.status == kv.KV_ERR_INVALID_ARG, bad
    # a bf16 latent pool holds rows (appends, handoff source); attention over
    # it is refused (no workspace size: the shape is unsupported)
    lat16 = kv.kv_pool_create(_desc(kv, layout=1, num_kv_heads=1, head_dim_k=576,
                                    head_dim_v=512, page_size=64, dtype=kv.KV_DTYPE_BF16,
                                    k_scale=None, v_cache=None, v_scale=None))
    assert kv._lib.paged_decode_workspace_size(lat16, 4, 16, 4) == 0
    kv.kv_pool_destroy(lat16)
    bf = _desc(kv, dtype=kv.KV_DTYPE_BF16, k_scale=None, v_scale=None)
    kv.kv_pool_destroy(kv.kv_pool_create(bf))


def test_handoff_argument_checks(kv):
    """kv_append_from_pool refuses bad arguments before enqueuing anything."""
    dst = kv.kv_pool_create(_desc(kv))
    src = kv.kv_pool_create(_desc(kv, dtype=kv.KV_DTYPE_BF16, k_scale=None, v_scale=None))
    src8 = kv.kv_pool_create(_desc(kv))  # an e4m3 source is refused
    other = kv.kv_pool_create(_desc(kv, dtype=kv.KV_DTYPE_BF16, k_scale=None, v_scale=None,
                                    page_size=32))
    f = 0x10000
    h = kv._lib.kv_append_from_pool
    bad = kv.KV_ERR_INVALID_ARG
    try:
        assert h(None, None, 2, src, f, 8, f, f, f, 8, f) == bad
        assert h(dst, None, 2, None, f, 8, f, f, f, 8, f) == bad
        assert h(dst, None, -1, src, f, 8, f, f, f, 8, f) == bad
        assert h(dst, None, 2, src, f, 0, f, f, f, 8, f) == bad
        assert h(dst, None, 2, src, f, 8, f, f, f, 0, f) == bad
        assert h(dst, None, 2, src, None, 8, f, f, f, 8, f) == bad
        assert h(dst, None, 2, src, f, 8, None, f, f, 8, f) == bad
        assert h(dst, None, 2, src, f, 8, f, None, f, 8, f) == bad
        assert h(dst, None, 2, src8, f, 8, f, f, f, 8, f) == bad    # source not bf16
        assert h(dst, None, 2, other, f, 8, f, f, f, 8, f) == bad   # page sizes differ
        assert h(dst, None, 0, src, None, 8, None, None, None, 8, None) == kv.KV_OK
        assert h(dst, None, 20000, src, f, 8, f, f, f, 8, f) == kv.KV_ERR_UNSUPPORTED
    finally:
        for x in (dst, src, src8, other):
            kv.kv_pool_destroy(x)


def test_entry_points_reject_bad_arguments(kv):
    lib = kv._lib
    h = kv.kv_pool_create(_desc(kv))
    try:
        assert lib.kv_append_quantize(h, None, -1, None, None, None, 0, None, None, 4, None) == 1
        assert lib.kv_append_quantize(h, None, 2, None, None, None, 1, None, None, 4, None) == 1
        assert lib.kv_append_quantize(h, None, 0, None, None, None, 0, None, None, 4, None) == 0
        assert lib.kv_verify_tags(h, None, 3, None, None, 4, None, None) == 1
        assert lib.kv_verify_tags(h, None, 0, None, None, 4, None, None) == 0
        assert lib.paged_decode_attn(h, None, 2, 8, 1, None, None, 4, None, None, 1.0, None,
                                     None, 0) == 1
        assert lib.paged_decode_attn_split(h, None, 2, 8, 1, 0x10000, 0x10000, 4, 0x10000, None,
                                           float("nan"), 0x10000, 1 << 20) == 1
        # workspace must be 256-byte aligned
        assert lib.paged_decode_attn_combine(h, None, 2, 8, 1, None, 0x10000, 0x10010, 1 << 20) == 1
        assert lib.kv_pool_destroy(None) == 1
        assert kv.kv_status_string(4) == "KV_ERR_OUT_OF_PAGES"
        assert lib.kv_last_launch_count(h) == 0
    finally:
        kv.kv_pool_destroy(h)


def test_release_argument_checks(kv):
    """kv_release_pages refuses bad arguments before enqueuing anything."""
    h = kv.kv_pool_create(_desc(kv))
    lib = kv._lib
    fake, ws = 0x10000, 0x20000
    need = kv.kv_release_workspace_size(4)
    assert need >= 8 * 5 and kv.kv_release_workspace_size(-1) == 0
    try:
        rel = lib.kv_release_pages
        assert rel(None, None, 4, fake, fake, 8, fake, None, ws, need) == kv.KV_ERR_INVALID_ARG
        assert rel(h, None, -1, fake, fake, 8, fake, None, ws, need) == kv.KV_ERR_INVALID_ARG
        assert rel(h, None, 4, fake, fake, 0, fake, None, ws, need) == kv.KV_ERR_INVALID_ARG
        assert rel(h, None, 4, None, fake, 8, fake, None, ws, need) == kv.KV_ERR_INVALID_ARG
        assert rel(h, None, 4, fake, fake, 8, fake, None, None, need) == kv.KV_ERR_INVALID_ARG
        assert rel(h, None, 4, fake, fake, 8, fake, None, ws + 4, need) == kv.KV_ERR_INVALID_ARG
        assert rel(h, None, 4, fake, fake, 8, fake, None, ws, need - 8) == kv.KV_ERR_INVALID_ARG
        assert rel(h, None, 0, None, None, 8, None, None, None, 0) == kv.KV_OK  # nothing to do
        assert kv.kv_status_string(kv.KV_ERR_TAG_MISMATCH) == "KV_ERR_TAG_MISMATCH"
    finally:
        kv.kv_pool_destroy(h)


def test_step_argument_checks(kv):
    """kv_decode_step refuses bad arguments before enqueuing anything (the
    checks below all come before any device query)."""
    h = kv.kv_pool_create(_desc(kv))
    lib = kv._lib
    f, ws = 0x10000, 0x20000
    assert kv.kv_decode_step_workspace_size(None, 4, 16, 1) == 0
    assert kv.kv_decode_step_workspace_size(h, -1, 16, 1) == 0
    try:
        def step(pool=h, B=4, flags=0, k=f, v=f, ind=f, max_new=1, pt=f, mp=8, sl=f, mask=f):
            return lib.kv_decode_step(pool, None, B, 16, 1, None, k, v, ind, max_new, pt, f, mp,
                                      sl, f, 1.0, f, mask, flags, ws, 1 << 20)
        bad = kv.KV_ERR_INVALID_ARG
        assert step(pool=None) == bad
        assert step(B=-1) == bad
        assert step(flags=2) == bad               # unknown flag bit
        assert step(max_new=-1) == bad
        assert step(mp=0) == bad
        assert step(mask=None) == bad             # the abort mask is always written
        assert step(ind=None) == bad
        assert step(pt=None) == bad
        assert step(sl=None) == bad
        assert step(k=None) == bad
        assert step(k=f + 2) == bad               # rows must be 16-byte aligned
        assert step(v=None) == bad                # GQA needs V rows
        assert step(B=0, mask=None, ind=None, pt=None, sl=None) == kv.KV_OK
        assert lib.kv_last_launch_count(h) == 0
    finally:
        kv.kv_pool_destroy(h)
