"""CPU oracle for the paged FP8 KV cache decode path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library in
``paged_fp8_kv_append_gb300`` never imports it and shares no code with it.

The arithmetic lives in ``kvfp8_oracle.c`` (plain single-threaded C, fp64
attention, exact e4m3 codec); this module compiles it with gcc and exposes
each entry point as a numpy-in, numpy-out function.  Every function keeps the
argument order of its C counterpart; see the C file for the definitions and
their sources.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvfp8_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, ERR_INVALID_ARG, ERR_OUT_OF_PAGES, ERR_BAD_PAGE_ID, ERR_TAG_MISMATCH = 0, 1, 4, 5, 8
# abort-mask bits of a step: the page-tag check failed / the append stopped first
ABORT_TAG, ABORT_UNSERVED = 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle (gcc -O2, no FMA contraction, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = [
            "gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm",
        ]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            vp, i32, u32, f32, i64 = (
                ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32, ctypes.c_float,
                ctypes.c_int64,
            )
            lib.or_e4m3_decode.argtypes = [u32]
            lib.or_e4m3_decode.restype = ctypes.c_double
            lib.or_e4m3_encode.argtypes = [f32]
            lib.or_e4m3_encode.restype = u32
            lib.or_e4m3_encode_bits_range.argtypes = [u32, u32, vp]
            lib.or_e4m3_encode_array.argtypes = [vp, i64, vp]
            lib.or_scale_from_amax.argtypes = [f32]
            lib.or_scale_from_amax.restype = f32
            lib.or_quantize.argtypes = [f32, f32]
            lib.or_quantize.restype = u32
            lib.or_alloc.argtypes = [i32, i32, vp, vp, vp, i32, vp, i32, vp, vp, i32, vp, vp, vp]
            lib.or_alloc.restype = i32
            lib.or_append_gqa.argtypes = (
                [i32] * 6 + [vp] * 7 + [i32] + [vp, vp, vp, i32, vp, vp, i32, vp, vp, i32]
            )
            lib.or_append_gqa.restype = i32
            lib.or_append_latent.argtypes = (
                [i32, i32, i32, i32] + [vp] * 5 + [i32, vp, vp, i32, vp, vp, i32, vp, vp, i32]
            )
            lib.or_append_latent.restype = i32
            lib.or_verify.argtypes = [i32, i32, vp, i32, vp, vp, i32, vp, vp]
            lib.or_release.argtypes = [i32, vp, vp, i32, vp, vp, i32, vp, vp]
            lib.or_release.restype = i32
            lib.or_attn_gqa.argtypes = (
                [i32] * 6 + [vp] * 4 + [i32, i32, i32, vp, i32, vp, vp, vp, f32, vp, vp]
            )
            lib.or_attn_latent.argtypes = (
                [i32] * 4 + [vp, vp] + [i32, i32, i32, vp, i32, vp, vp, vp, f32, vp, vp]
            )
            _lib = lib
    return _lib


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags.c_contiguous, "oracle wants C-contiguous numpy"
    return a.ctypes.data_as(ctypes.c_void_p)


# -- codec -----------------------------------------------------------------

def e4m3_decode(code: int) -> float:
    return _load().or_e4m3_decode(int(code))


def e4m3_encode(x: float) -> int:
    return int(_load().or_e4m3_encode(float(x)))


def e4m3_encode_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().or_e4m3_encode_array(_p(x), x.size, _p(out))
    return out


def e4m3_encode_bits_range(first: int, count: int) -> np.ndarray:
    out = np.empty(count, dtype=np.uint8)
    _load().or_e4m3_encode_bits_range(first, count, _p(out))
    return out


def scale_from_amax(amax: float) -> float:
    return float(_load().or_scale_from_amax(float(amax)))


# -- pool state ------------------------------------------------------------

class Pool:
    """Host copy of a pool's buffers, laid out as the library documents them.

    GQA:    k_cache[page][kv_head][slot][dk], v_cache[page][kv_head][dv][slot]
    LATENT: k_cache[page][slot][dk] (v_cache unused), one scale per page.
    e4m3 caches are uint8; bf16 caches are uint16 bit patterns.
    """

    def __init__(self, num_pages, page_size, num_kv_heads, dk, dv, dtype=0,
                 layout=0, tags=None, free_list=None, scale_mode=0):
        self.num_pages, self.page_size = int(num_pages), int(page_size)
        self.scale_mode = int(scale_mode)  # 0: frozen scales; 1: re-quantise
        self.num_kv_heads, self.dk, self.dv = int(num_kv_heads), int(dk), int(dv)
        self.dtype, self.layout = int(dtype), int(layout)
        edt = np.uint8 if dtype == 0 else np.uint16
        if layout == 0:
            self.k_cache = np.zeros((num_pages, num_kv_heads, page_size, dk), edt)
            self.v_cache = np.zeros((num_pages, num_kv_heads, dv, page_size), edt)
            self.k_scale = np.zeros((num_pages, num_kv_heads), np.float32)
            self.v_scale = np.zeros((num_pages, num_kv_heads), np.float32)
        else:
            assert num_kv_heads == 1
            self.k_cache = np.zeros((num_pages, page_size, dk), edt)
            self.v_cache = None
            self.k_scale = np.zeros((num_pages,), np.float32)
            self.v_scale = None
        self.tags = (np.zeros(num_pages, np.uint32) if tags is None
                     else np.array(tags, dtype=np.uint32))
        self.free_list = (np.arange(num_pages, dtype=np.int32) if free_list is None
                          else np.array(free_list, dtype=np.int32))
        self.free_head = np.zeros(1, np.int32)


def alloc(pool: Pool, new_indptr, max_new, page_table, exp_tags, seq_lens):
    """Bookkeeping only (page pops, tag stamps); returns (status, stop_req)."""
    B = len(seq_lens)
    stop = np.zeros(1, np.int32)
    st = _load().or_alloc(pool.num_pages, pool.page_size, _p(pool.tags), _p(pool.free_list),
                          _p(pool.free_head), B, _p(new_indptr), int(max_new), _p(page_table),
                          _p(exp_tags), page_table.shape[1], _p(seq_lens), _p(stop), None)
    return int(st), int(stop[0])


def append(pool: Pool, k_new, v_new, new_indptr, max_new, page_table, exp_tags, seq_lens):
    """Append (quantise-on-write for e4m3).  Arrays are updated in place.

    k_new / v_new: uint16 bf16 bit patterns [rows][kv_heads][d] (GQA) or
    [rows][dk] (latent; v_new ignored).  Returns (status, stop_req).
    """
    B = len(seq_lens)
    stop = np.zeros(1, np.int32)
    new_indptr = np.ascontiguousarray(new_indptr, np.int32)
    lib = _load()
    if pool.layout == 0:
        st = lib.or_append_gqa(
            pool.num_pages, pool.page_size, pool.num_kv_heads, pool.dk, pool.dv, pool.dtype,
            _p(pool.k_cache), _p(pool.v_cache), _p(pool.k_scale), _p(pool.v_scale),
            _p(pool.tags), _p(pool.free_list), _p(pool.free_head), B,
            _p(np.ascontiguousarray(k_new, np.uint16)), _p(np.ascontiguousarray(v_new, np.uint16)),
            _p(new_indptr), int(max_new), _p(page_table), _p(exp_tags), page_table.shape[1],
            _p(seq_lens), _p(stop), pool.scale_mode)
    else:
        st = lib.or_append_latent(
            pool.num_pages, pool.page_size, pool.dk, pool.dtype, _p(pool.k_cache),
            _p(pool.k_scale),
            _p(pool.tags), _p(pool.free_list), _p(pool.free_head), B,
            _p(np.ascontiguousarray(k_new, np.uint16)), _p(new_indptr), int(max_new),
            _p(page_table), _p(exp_tags), page_table.shape[1], _p(seq_lens), _p(stop),
            pool.scale_mode)
    return int(st), int(stop[0])


def release(pool: Pool, page_table, exp_tags, seq_lens, mask=None):
    """Return the pages of the masked requests (all when mask is None) to the
    free list.  Arrays are updated in place; returns the status."""
    B = len(seq_lens)
    m = None if mask is None else np.ascontiguousarray(mask, np.uint8)
    return int(_load().or_release(pool.page_size, _p(pool.free_list), _p(pool.free_head), B,
                                  _p(page_table), _p(exp_tags), page_table.shape[1],
                                  _p(seq_lens), _p(m)))


def verify(pool_num_pages, page_size, tags, page_table, exp_tags, seq_lens):
    B = len(seq_lens)
    mask = np.zeros(B, np.uint8)
    _load().or_verify(int(pool_num_pages), int(page_size),
                      _p(np.ascontiguousarray(tags, np.uint32)), B,
                      _p(np.ascontiguousarray(page_table, np.int32)),
                      _p(np.ascontiguousarray(exp_tags, np.uint32)), page_table.shape[1],
                      _p(np.ascontiguousarray(seq_lens, np.int32)), _p(mask))
    return mask


def attn(pool: Pool, q_bits, page_table, seq_lens, abort_mask, sm_scale, num_q_heads, q_tokens):
    """fp64 decode attention.  q_bits: uint16 bf16 [B][T][Hq][dk].

    Returns (out fp64 [B][T][Hq][dv], written uint8 [B]).
    """
    B = len(seq_lens)
    T, Hq = int(q_tokens), int(num_q_heads)
    q_bits = np.ascontiguousarray(q_bits, np.uint16)
    assert q_bits.shape == (B, T, Hq, pool.dk)
    out = np.zeros((B, T, Hq, pool.dv), np.float64)
    written = np.zeros(B, np.uint8)
    pt = np.ascontiguousarray(page_table, np.int32)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    am = None if abort_mask is None else np.ascontiguousarray(abort_mask, np.uint8)
    lib = _load()
    if pool.layout == 0:
        lib.or_attn_gqa(pool.num_pages, pool.page_size, pool.num_kv_heads, pool.dk, pool.dv,
                        pool.dtype, _p(pool.k_cache), _p(pool.v_cache),
                        _p(pool.k_scale) if pool.dtype == 0 else None,
                        _p(pool.v_scale) if pool.dtype == 0 else None,
                        B, Hq, T, _p(pt), pt.shape[1], _p(sl), _p(am), _p(q_bits),
                        float(np.float32(sm_scale)), _p(out), _p(written))
    else:
        assert pool.dtype == 0, "latent attention reads an e4m3 pool"
        lib.or_attn_latent(pool.num_pages, pool.page_size, pool.dk, pool.dv,
                           _p(pool.k_cache), _p(pool.k_scale), B, Hq, T, _p(pt), pt.shape[1],
                           _p(sl), _p(am), _p(q_bits), float(np.float32(sm_scale)), _p(out),
                           _p(written))
    return out, written


def step(pool: Pool, leave_mask, k_new, v_new, new_indptr, max_new, page_table, exp_tags,
         seq_lens, q_bits, sm_scale, num_q_heads, q_tokens, remove_aborted=True):
    """One continuous-batching decode step over B request slots ("Smaller,
    faster, safer: running Kimi and GLM at scale", section "Protecting a
    shared KV cache": the tag check runs on every step, before attention, and
    a request that fails it is aborted and returns no data).  A slot with
    length 0 is empty.  In order:

    1. requests with leave_mask[r] != 0 release their pages (release());
    2. the tag check over every mapping that exists now: abort bit ABORT_TAG;
    3. the append, in which a request with ABORT_TAG appends nothing (its
       rows are dropped); every request at or after the append's stop index
       gets ABORT_UNSERVED;
    4. attention for every request whose abort mask is 0;
    5. with remove_aborted, requests with ABORT_TAG release their pages.

    The mappings the append creates are pages it has just popped, with the
    tag it has just stamped, and the rows it puts into a partly filled page
    go there only after step 2 found that page's tag unchanged; so every
    page attention reads has passed the check.  Arrays are updated in place.
    Returns (status, abort_mask, out, written); status is the first nonzero
    status of the phases."""
    status = OK
    if leave_mask is not None:
        status = release(pool, page_table, exp_tags, seq_lens, leave_mask)
    mask = verify(pool.num_pages, pool.page_size, pool.tags, page_table, exp_tags, seq_lens)
    ind = np.asarray(new_indptr, np.int64)
    B = len(seq_lens)
    keep = [r for r in range(B) if not mask[r]]
    counts = np.zeros(B, np.int64)
    counts[keep] = ind[1:][keep] - ind[:-1][keep]
    ind_eff = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    k_new = np.asarray(k_new)
    ks = [k_new[ind[r]:ind[r + 1]] for r in keep]
    k_eff = np.concatenate(ks) if ks else k_new[:0]
    v_eff = None
    if v_new is not None:
        v_new = np.asarray(v_new)
        vs = [v_new[ind[r]:ind[r + 1]] for r in keep]
        v_eff = np.concatenate(vs) if vs else v_new[:0]
    st, stop = append(pool, k_eff, v_eff if v_eff is not None else k_eff, ind_eff, max_new,
                      page_table, exp_tags, seq_lens)
    status = status or st
    mask[stop:] |= ABORT_UNSERVED
    out, written = attn(pool, q_bits, page_table, seq_lens, mask, sm_scale, num_q_heads,
                        q_tokens)
    if remove_aborted:
        stale = (mask & ABORT_TAG).astype(np.uint8)
        if stale.any():
            # runs whatever an earlier phase reported; the first error is kept
            st = release(pool, page_table, exp_tags, seq_lens, stale)
            status = status or st
    return status, mask, out, written
