"""Python binding of the GB300 paged FP8 KV cache library (include/kvfp8.h).

Argument marshalling only: every function takes torch tensors (device
memory) and forwards their pointers to the C ABI in ``libkvfp8.so``; all
compute runs in the library's CUDA kernels.  Importing this package raises if
the library has not been built (``python -m paged_fp8_kv_append_gb300.build``
or ``__graft_entry__.build()``): there is no fallback path.

The method follows "Smaller, faster, safer: running Kimi and GLM at scale"
(sections "Quantizing the KV cache" and "Protecting a shared KV cache").
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvfp8.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python -m paged_fp8_kv_append_gb300.build)")

_lib = ctypes.CDLL(LIB_PATH)

# status codes
KV_OK, KV_ERR_INVALID_ARG, KV_ERR_UNSUPPORTED, KV_ERR_CUDA = 0, 1, 2, 3
KV_ERR_OUT_OF_PAGES, KV_ERR_BAD_PAGE_ID, KV_ERR_TIMEOUT, KV_ERR_INTERNAL = 4, 5, 6, 7
KV_ERR_TAG_MISMATCH = 8
KV_DTYPE_E4M3, KV_DTYPE_BF16 = 0, 1
KV_LAYOUT_GQA, KV_LAYOUT_LATENT = 0, 1
KV_SCALE_FROZEN, KV_SCALE_REQUANTIZE = 0, 1
KV_ABORT_TAG, KV_ABORT_UNSERVED, KV_STEP_REMOVE_ABORTED = 1, 2, 1
KV_CTL_FREE_HEAD, KV_CTL_ERROR, KV_CTL_APPEND_STOP, KV_CTL_WAIT_INFO, KV_CTL_WORDS = 0, 1, 2, 3, 4


class kv_pool_desc(ctypes.Structure):
    _fields_ = [
        ("num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim_k", ctypes.c_int32),
        ("head_dim_v", ctypes.c_int32), ("dtype", ctypes.c_int32), ("layout", ctypes.c_int32),
        ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
        ("tags", ctypes.c_void_p), ("free_list", ctypes.c_void_p), ("ctl", ctypes.c_void_p),
        ("scale_mode", ctypes.c_int32),
    ]


_vp, _i32, _f32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
_lib.kv_pool_create.argtypes = [ctypes.POINTER(kv_pool_desc), ctypes.POINTER(_vp)]
_lib.kv_pool_create.restype = _i32
_lib.kv_pool_destroy.argtypes = [_vp]
_lib.kv_pool_destroy.restype = _i32
_lib.kv_append_quantize.argtypes = [_vp, _vp, _i32, _vp, _vp, _vp, _i32, _vp, _vp, _i32, _vp]
_lib.kv_append_quantize.restype = _i32
_lib.kv_append_from_pool.argtypes = [_vp, _vp, _i32, _vp, _vp, _i32, _vp, _vp, _vp, _i32, _vp]
_lib.kv_append_from_pool.restype = _i32
_lib.kv_verify_tags.argtypes = [_vp, _vp, _i32, _vp, _vp, _i32, _vp, _vp]
_lib.kv_verify_tags.restype = _i32
_lib.kv_release_workspace_size.argtypes = [_i32]
_lib.kv_release_workspace_size.restype = _sz
_lib.kv_release_pages.argtypes = [_vp, _vp, _i32, _vp, _vp, _i32, _vp, _vp, _vp, _sz]
_lib.kv_release_pages.restype = _i32
_lib.paged_decode_workspace_size.argtypes = [_vp, _i32, _i32, _i32]
_lib.paged_decode_workspace_size.restype = _sz
_lib.paged_decode_attn.argtypes = [_vp, _vp, _i32, _i32, _i32, _vp, _vp, _i32, _vp, _vp, _f32,
                                   _vp, _vp, _sz]
_lib.paged_decode_attn.restype = _i32
_lib.paged_decode_attn_split.argtypes = [_vp, _vp, _i32, _i32, _i32, _vp, _vp, _i32, _vp, _vp,
                                         _f32, _vp, _sz]
_lib.paged_decode_attn_split.restype = _i32
_lib.paged_decode_attn_combine.argtypes = [_vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _sz]
_lib.paged_decode_attn_combine.restype = _i32
_lib.paged_decode_attn_checked.argtypes = [_vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _i32, _vp,
                                           _f32, _vp, _vp, _vp, _sz]
_lib.paged_decode_attn_checked.restype = _i32
_lib.paged_decode_attn_noalloc.argtypes = [_vp, _vp, _i32, _i32, _i32, _vp, _vp, _i32, _vp,
                                           _vp, _f32, _vp]
_lib.paged_decode_attn_noalloc.restype = _i32
_lib.kv_decode_step_workspace_size.argtypes = [_vp, _i32, _i32, _i32]
_lib.kv_decode_step_workspace_size.restype = _sz
_lib.kv_decode_step.argtypes = [_vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _i32, _vp, _vp,
                                _i32, _vp, _vp, _f32, _vp, _vp, _i32, _vp, _sz]
_lib.kv_decode_step.restype = _i32
_lib.kv_status_string.argtypes = [_i32]
_lib.kv_status_string.restype = ctypes.c_char_p
_lib.kv_last_launch_count.argtypes = [_vp]
_lib.kv_last_launch_count.restype = _i32


def u32_as_i32(a) -> torch.Tensor:
    """uint32 values (numpy / list / tensor) as an int32 tensor with the same bits."""
    import numpy as np

    if isinstance(a, torch.Tensor):
        return a.view(torch.int32) if a.dtype == torch.uint32 else a.to(torch.int32)
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.uint32)).view(np.int32))


class KVError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {kv_status_string(status)}")


def kv_status_string(status: int) -> str:
    return _lib.kv_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != KV_OK:
        raise KVError(status, where)


_U32 = (torch.int32, torch.uint32)  # uint32 arrays may be held as int32 (same bits)


def _ptr(t, dtype=None, name="tensor"):
    """Device pointer of a contiguous CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    allowed = dtype if isinstance(dtype, tuple) else (dtype,)
    if dtype is not None and t.dtype not in allowed:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream)


# ---------------------------------------------------------------- raw C ABI

def kv_pool_create(desc: kv_pool_desc) -> int:
    h = _vp()
    _check(_lib.kv_pool_create(ctypes.byref(desc), ctypes.byref(h)), "kv_pool_create")
    return h.value


def kv_pool_destroy(handle: int) -> None:
    _check(_lib.kv_pool_destroy(handle), "kv_pool_destroy")


def kv_last_launch_count(handle: int) -> int:
    return int(_lib.kv_last_launch_count(handle))


def kv_append_quantize(handle, B, k_new, v_new, new_indptr, max_new_per_req, page_table,
                       exp_tags, seq_lens, stream=None):
    st = _lib.kv_append_quantize(
        handle, _stream(stream), int(B), _ptr(k_new, torch.bfloat16, "k_new"),
        _ptr(v_new, torch.bfloat16, "v_new"), _ptr(new_indptr, torch.int32, "new_indptr"),
        int(max_new_per_req), _ptr(page_table, torch.int32, "page_table"),
        _ptr(exp_tags, _U32, "exp_tags"), int(page_table.shape[-1]),
        _ptr(seq_lens, torch.int32, "seq_lens"))
    _check(st, "kv_append_quantize")


def kv_append_from_pool(handle, B, src_handle, src_page_table, src_seq_lens, page_table,
                        exp_tags, seq_lens, stream=None):
    """Append each request's rows of a bf16 source pool (read through its page
    table) to this pool, as kv_append_quantize would (see kvfp8.h)."""
    st = _lib.kv_append_from_pool(
        handle, _stream(stream), int(B), src_handle,
        _ptr(src_page_table, torch.int32, "src_page_table"), int(src_page_table.shape[-1]),
        _ptr(src_seq_lens, torch.int32, "src_seq_lens"),
        _ptr(page_table, torch.int32, "page_table"), _ptr(exp_tags, _U32, "exp_tags"),
        int(page_table.shape[-1]), _ptr(seq_lens, torch.int32, "seq_lens"))
    _check(st, "kv_append_from_pool")


def kv_verify_tags(handle, B, page_table, exp_tags, seq_lens, abort_mask, stream=None):
    st = _lib.kv_verify_tags(
        handle, _stream(stream), int(B), _ptr(page_table, torch.int32, "page_table"),
        _ptr(exp_tags, _U32, "exp_tags"), int(page_table.shape[-1]),
        _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(abort_mask, torch.uint8, "abort_mask"))
    _check(st, "kv_verify_tags")


def kv_release_workspace_size(B) -> int:
    return int(_lib.kv_release_workspace_size(int(B)))


def kv_release_pages(handle, B, page_table, exp_tags, seq_lens, release_mask, workspace,
                     stream=None):
    st = _lib.kv_release_pages(
        handle, _stream(stream), int(B), _ptr(page_table, torch.int32, "page_table"),
        _ptr(exp_tags, _U32, "exp_tags"), int(page_table.shape[-1]),
        _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(release_mask, torch.uint8, "release_mask"),
        _ptr(workspace, torch.uint8, "workspace"), int(workspace.numel()))
    _check(st, "kv_release_pages")


def paged_decode_workspace_size(handle, B, num_q_heads, q_tokens) -> int:
    return int(_lib.paged_decode_workspace_size(handle, int(B), int(num_q_heads), int(q_tokens)))


def paged_decode_attn(handle, B, num_q_heads, q_tokens, q, page_table, seq_lens, abort_mask,
                      sm_scale, out, workspace, stream=None):
    st = _lib.paged_decode_attn(
        handle, _stream(stream), int(B), int(num_q_heads), int(q_tokens),
        _ptr(q, torch.bfloat16, "q"), _ptr(page_table, torch.int32, "page_table"),
        int(page_table.shape[-1]), _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(abort_mask, torch.uint8, "abort_mask"), float(sm_scale),
        _ptr(out, torch.bfloat16, "out"), _ptr(workspace, torch.uint8, "workspace"),
        int(workspace.numel()))
    _check(st, "paged_decode_attn")


def paged_decode_attn_checked(handle, B, num_q_heads, q_tokens, q, page_table, exp_tags,
                              seq_lens, sm_scale, out, abort_mask, workspace, stream=None):
    """paged_decode_attn with the page-tag check fused into the page reads;
    writes abort_mask (see kvfp8.h)."""
    st = _lib.paged_decode_attn_checked(
        handle, _stream(stream), int(B), int(num_q_heads), int(q_tokens),
        _ptr(q, torch.bfloat16, "q"), _ptr(page_table, torch.int32, "page_table"),
        _ptr(exp_tags, _U32, "exp_tags"), int(page_table.shape[-1]),
        _ptr(seq_lens, torch.int32, "seq_lens"), float(sm_scale),
        _ptr(out, torch.bfloat16, "out"), _ptr(abort_mask, torch.uint8, "abort_mask"),
        _ptr(workspace, torch.uint8, "workspace"), int(workspace.numel()))
    _check(st, "paged_decode_attn_checked")


def paged_decode_attn_noalloc(handle, B, num_q_heads, q_tokens, q, page_table, seq_lens,
                              abort_mask, sm_scale, out, stream=None):
    """paged_decode_attn with the library's fixed device scratch instead of a
    workspace: for callers that cannot allocate device memory (see kvfp8.h)."""
    st = _lib.paged_decode_attn_noalloc(
        handle, _stream(stream), int(B), int(num_q_heads), int(q_tokens),
        _ptr(q, torch.bfloat16, "q"), _ptr(page_table, torch.int32, "page_table"),
        int(page_table.shape[-1]), _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(abort_mask, torch.uint8, "abort_mask"), float(sm_scale),
        _ptr(out, torch.bfloat16, "out"))
    _check(st, "paged_decode_attn_noalloc")


def paged_decode_attn_split(handle, B, num_q_heads, q_tokens, q, page_table, seq_lens,
                            abort_mask, sm_scale, workspace, stream=None):
    st = _lib.paged_decode_attn_split(
        handle, _stream(stream), int(B), int(num_q_heads), int(q_tokens),
        _ptr(q, torch.bfloat16, "q"), _ptr(page_table, torch.int32, "page_table"),
        int(page_table.shape[-1]), _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(abort_mask, torch.uint8, "abort_mask"), float(sm_scale),
        _ptr(workspace, torch.uint8, "workspace"), int(workspace.numel()))
    _check(st, "paged_decode_attn_split")


def paged_decode_attn_combine(handle, B, num_q_heads, q_tokens, abort_mask, out, workspace,
                              stream=None):
    st = _lib.paged_decode_attn_combine(
        handle, _stream(stream), int(B), int(num_q_heads), int(q_tokens),
        _ptr(abort_mask, torch.uint8, "abort_mask"), _ptr(out, torch.bfloat16, "out"),
        _ptr(workspace, torch.uint8, "workspace"), int(workspace.numel()))
    _check(st, "paged_decode_attn_combine")


def kv_decode_step_workspace_size(handle, B, num_q_heads, q_tokens) -> int:
    return int(_lib.kv_decode_step_workspace_size(handle, int(B), int(num_q_heads),
                                                  int(q_tokens)))


def kv_decode_step(handle, B, num_q_heads, q_tokens, leave_mask, k_new, v_new, new_indptr,
                   max_new_per_req, page_table, exp_tags, seq_lens, q, sm_scale, out, abort_mask,
                   flags, workspace, stream=None):
    st = _lib.kv_decode_step(
        handle, _stream(stream), int(B), int(num_q_heads), int(q_tokens),
        _ptr(leave_mask, torch.uint8, "leave_mask"), _ptr(k_new, torch.bfloat16, "k_new"),
        _ptr(v_new, torch.bfloat16, "v_new"), _ptr(new_indptr, torch.int32, "new_indptr"),
        int(max_new_per_req), _ptr(page_table, torch.int32, "page_table"),
        _ptr(exp_tags, _U32, "exp_tags"), int(page_table.shape[-1]),
        _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(q, torch.bfloat16, "q"), float(sm_scale),
        _ptr(out, torch.bfloat16, "out"), _ptr(abort_mask, torch.uint8, "abort_mask"),
        int(flags), _ptr(workspace, torch.uint8, "workspace"), int(workspace.numel()))
    _check(st, "kv_decode_step")


# ---------------------------------------------------------------- pool helper

class KVPool:
    """A pool whose buffers are torch tensors on one CUDA device.

    Allocates the caller-owned buffers the C ABI documents (cache, scales,
    tags, free list, control block) and holds the library handle.  GQA:
    k_cache [pages][Hkv][P][Dk], v_cache [pages][Hkv][Dv][P]; LATENT:
    k_cache [pages][P][Dk].  e4m3 caches are uint8 tensors.
    """

    def __init__(self, num_pages, page_size, num_kv_heads, head_dim_k, head_dim_v,
                 dtype=KV_DTYPE_E4M3, layout=KV_LAYOUT_GQA, device="cuda", tags=None,
                 free_list=None, scale_mode=KV_SCALE_FROZEN):
        dev = torch.device(device)
        self.scale_mode = int(scale_mode)
        self.num_pages, self.page_size = int(num_pages), int(page_size)
        self.num_kv_heads, self.head_dim_k, self.head_dim_v = (
            int(num_kv_heads), int(head_dim_k), int(head_dim_v))
        self.dtype, self.layout = int(dtype), int(layout)
        edt = torch.uint8 if dtype == KV_DTYPE_E4M3 else torch.bfloat16
        if layout == KV_LAYOUT_GQA:
            self.k_cache = torch.zeros((num_pages, num_kv_heads, page_size, head_dim_k), dtype=edt,
                                       device=dev)
            self.v_cache = torch.zeros((num_pages, num_kv_heads, head_dim_v, page_size), dtype=edt,
                                       device=dev)
            if dtype == KV_DTYPE_E4M3:
                self.k_scale = torch.zeros((num_pages, num_kv_heads), dtype=torch.float32, device=dev)
                self.v_scale = torch.zeros((num_pages, num_kv_heads), dtype=torch.float32, device=dev)
            else:
                self.k_scale = self.v_scale = None
        else:
            self.k_cache = torch.zeros((num_pages, page_size, head_dim_k), dtype=edt, device=dev)
            self.v_cache = None
            self.k_scale = (torch.zeros((num_pages,), dtype=torch.float32, device=dev)
                            if dtype == KV_DTYPE_E4M3 else None)
            self.v_scale = None
        # uint32 tags held in an int32 tensor (same bits; torch has few uint32 ops)
        self.tags = (torch.zeros(num_pages, dtype=torch.int32, device=dev) if tags is None
                     else u32_as_i32(tags).to(dev))
        self.free_list = (torch.arange(num_pages, dtype=torch.int32, device=dev) if free_list is None
                          else torch.as_tensor(free_list, dtype=torch.int32).to(dev))
        self.ctl = torch.zeros(KV_CTL_WORDS, dtype=torch.int32, device=dev)
        d = kv_pool_desc()
        d.num_pages, d.page_size, d.num_kv_heads = self.num_pages, self.page_size, self.num_kv_heads
        d.head_dim_k, d.head_dim_v, d.dtype, d.layout = (
            self.head_dim_k, self.head_dim_v, self.dtype, self.layout)
        d.k_cache = self.k_cache.data_ptr()
        d.v_cache = self.v_cache.data_ptr() if self.v_cache is not None else None
        d.k_scale = self.k_scale.data_ptr() if self.k_scale is not None else None
        d.v_scale = self.v_scale.data_ptr() if self.v_scale is not None else None
        d.tags, d.free_list, d.ctl = (self.tags.data_ptr(), self.free_list.data_ptr(),
                                      self.ctl.data_ptr())
        d.scale_mode = self.scale_mode
        self.desc = d
        self.handle = kv_pool_create(d)

    def close(self):
        if getattr(self, "handle", None):
            kv_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # convenience wrappers (same argument order as the C ABI)
    def append(self, B, k_new, v_new, new_indptr, max_new_per_req, page_table, exp_tags,
               seq_lens, stream=None):
        kv_append_quantize(self.handle, B, k_new, v_new, new_indptr, max_new_per_req,
                           page_table, exp_tags, seq_lens, stream)

    def append_from_pool(self, B, src, src_page_table, src_seq_lens, page_table, exp_tags,
                         seq_lens, stream=None):
        kv_append_from_pool(self.handle, B, src.handle, src_page_table, src_seq_lens, page_table,
                            exp_tags, seq_lens, stream)

    def verify(self, B, page_table, exp_tags, seq_lens, abort_mask, stream=None):
        kv_verify_tags(self.handle, B, page_table, exp_tags, seq_lens, abort_mask, stream)

    def release(self, B, page_table, exp_tags, seq_lens, release_mask, workspace, stream=None):
        kv_release_pages(self.handle, B, page_table, exp_tags, seq_lens, release_mask, workspace,
                         stream)

    def workspace_size(self, B, num_q_heads, q_tokens) -> int:
        n = paged_decode_workspace_size(self.handle, B, num_q_heads, q_tokens)
        if n == 0 and B > 0:
            raise KVError(KV_ERR_UNSUPPORTED, "paged_decode_workspace_size")
        return n

    def attn(self, B, num_q_heads, q_tokens, q, page_table, seq_lens, abort_mask, sm_scale, out,
             workspace, stream=None):
        paged_decode_attn(self.handle, B, num_q_heads, q_tokens, q, page_table, seq_lens,
                          abort_mask, sm_scale, out, workspace, stream)

    def step_workspace_size(self, B, num_q_heads, q_tokens) -> int:
        n = kv_decode_step_workspace_size(self.handle, B, num_q_heads, q_tokens)
        if n == 0 and B > 0:
            raise KVError(KV_ERR_UNSUPPORTED, "kv_decode_step_workspace_size")
        return n

    def step(self, B, num_q_heads, q_tokens, leave_mask, k_new, v_new, new_indptr,
             max_new_per_req, page_table, exp_tags, seq_lens, q, sm_scale, out, abort_mask,
             flags, workspace, stream=None):
        kv_decode_step(self.handle, B, num_q_heads, q_tokens, leave_mask, k_new, v_new,
                       new_indptr, max_new_per_req, page_table, exp_tags, seq_lens, q, sm_scale,
                       out, abort_mask, flags, workspace, stream)

    def error(self) -> int:
        """Device error word (synchronises)."""
        return int(self.ctl[KV_CTL_ERROR].item())

    def launches(self) -> int:
        return kv_last_launch_count(self.handle)
