"""ctypes binding of libcpattn: torch tensors in, C-ABI calls out.

Argument marshalling only -- every step of the computation runs in the CUDA
library.  There is no fallback: if ``libcpattn.so`` is missing or fails to
load, every call raises.  Tensors must be CUDA, contiguous and of the
documented dtype; the current torch stream is used unless one is given.
"""

from __future__ import annotations

import ctypes
import os

import torch

from .build_lib import LIB

DTYPE_BF16 = 0
DTYPE_FP32 = 1
DTYPE_FP8_E4M3 = 2  # pools only
FP8_NAN_CODE = 0x7F
LSE_TOKEN_MAJOR = 0
LSE_HEAD_MAJOR = 1
MAX_MERGE_VIEWS = 16

_STATUS_NAMES = {
    0: "CPATTN_OK",
    -1: "CPATTN_ERR_INVALID_ARG",
    -2: "CPATTN_ERR_P_NOT_DIVIDING_PAGE_SIZE",
    -3: "CPATTN_ERR_UNSUPPORTED_SHAPE",
    -4: "CPATTN_ERR_MISALIGNED",
    -5: "CPATTN_ERR_WORKSPACE_TOO_SMALL",
    -6: "CPATTN_ERR_CUDA",
}


class CpattnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what} failed: {_STATUS_NAMES.get(status, status)} ({status})")


class PoolDesc(ctypes.Structure):
    """Mirror of ``cpattn_pool_desc``."""

    _fields_ = [
        ("P", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("head_dim_v", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("interleave", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
        ("k_descale", ctypes.c_float),
        ("v_descale", ctypes.c_float),
    ]

    @property
    def mla(self) -> bool:
        return self.head_dim_v != self.head_dim

    def pool_shape(self, value: bool = False):
        d = self.head_dim_v if value else self.head_dim
        return (self.P, self.num_pages, self.num_kv_heads, self.page_size // self.P, d)

    def torch_dtype(self):
        """Type of queries, new K/V and outputs."""
        return torch.bfloat16 if self.dtype == DTYPE_BF16 else torch.float32

    @property
    def fp8(self) -> bool:
        return self.kv_dtype == DTYPE_FP8_E4M3

    def pool_torch_dtype(self):
        """Element type of pool_k / pool_v tensors (E4M3 codes as uint8)."""
        return torch.uint8 if self.fp8 else self.torch_dtype()


class PartialView(ctypes.Structure):
    """Mirror of ``cpattn_partial_view``."""

    _fields_ = [
        ("o", ctypes.c_void_p),
        ("lse", ctypes.c_void_p),
        ("o_stride_token", ctypes.c_int64),
        ("o_stride_head", ctypes.c_int64),
        ("lse_stride_token", ctypes.c_int64),
        ("lse_stride_head", ctypes.c_int64),
    ]


_lib = None
_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t
_f32 = ctypes.c_float
_pdesc = ctypes.POINTER(PoolDesc)

_SIGNATURES = {
    "cpattn_version": (_i32, []),
    "cpattn_status_string": (ctypes.c_char_p, [_i32]),
    "cpattn_pool_bytes": (_sz, [_pdesc, _i32]),
    "cp_kv_write": (_i32, [_pdesc, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp]),
    "cp_paged_attn_partial": (_i32, [_pdesc, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _i32, _vp, _vp, _f32,
                                     _vp, _vp, _vp, _sz, _vp, _vp]),
    "cp_paged_attn_workspace_bytes": (_sz, [_pdesc, _i32, _i32, _i32]),
    "cp_paged_attn_partial_ex": (_i32, [_pdesc, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _i32, _vp, _vp, _f32,
                                        _vp, _vp, _i32, _vp, _vp, _sz, _vp, _vp]),
    "lse_merge_views": (_i32, [_i32, ctypes.POINTER(PartialView), _i32, _i32, _i32, _i32, _vp, _i64, _i64, _vp,
                               _i64, _i64, _vp]),
    "cp_paged_attn_fused": (_i32, [_pdesc, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _i32, _vp, _vp, _vp, _f32,
                                   _vp, _vp, _i32, _vp, _vp, _vp, _sz, _vp, _vp]),
    "cp_paged_attn_fused_workspace_bytes": (_sz, [_pdesc, _i32, _i32, _i32]),
    "own_token_attn": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _i32, _i32, _i32, _i32, _f32,
                              _vp, _vp, _vp]),
    "lse_merge": (_i32, [_i32, _vp, _vp, _i64, _i64, _i32, _i32, _i32, _i32, _vp, _vp, _vp]),
}


def library_path() -> str:
    return LIB


def load_library(path: str | None = None):
    """Load libcpattn.so (once).  Raises if it is missing: there is no fallback."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(p)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if lib.cpattn_version() != 3:
        raise RuntimeError("libcpattn version mismatch")
    if path is None:
        _lib = lib
    return lib


def version() -> int:
    return load_library().cpattn_version()


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _i32_tensor(t, what):
    if t is not None and t.dtype != torch.int32:
        raise TypeError(f"{what} must be int32")
    return _ptr(t)


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check(status, what):
    if status != 0:
        raise CpattnError(status, what)


def cp_kv_write(desc: PoolDesc, pool_k, pool_v, k_new, v_new, positions, qo_indptr, kv_page_indptr,
                kv_page_indices, dev_status=None, stream=None):
    """Write new K/V rows into the striped pool (see ``cp_kv_write`` in cpattn.h)."""
    lib = load_library()
    num_rows = qo_indptr.numel() - 1
    st = lib.cp_kv_write(ctypes.byref(desc), _ptr(pool_k), _ptr(pool_v), _ptr(k_new), _ptr(v_new),
                         _i32_tensor(positions, "positions"), _i32_tensor(qo_indptr, "qo_indptr"), num_rows,
                         positions.numel(), _i32_tensor(kv_page_indptr, "kv_page_indptr"),
                         _i32_tensor(kv_page_indices, "kv_page_indices"), _i32_tensor(dev_status, "dev_status"),
                         _stream(stream))
    _check(st, "cp_kv_write")


def workspace_bytes(desc: PoolDesc, num_q_heads: int, num_tokens: int, max_kv_len: int) -> int:
    return load_library().cp_paged_attn_workspace_bytes(ctypes.byref(desc), num_q_heads, num_tokens, max_kv_len)


def cp_paged_attn_partial(desc: PoolDesc, pool_k, pool_v, q, kv_len, max_kv_len, kv_page_indptr, kv_page_indices,
                          scale, o_part, lse_part, workspace, qo_indptr=None, num_rows=None, dev_status=None,
                          stream=None):
    """Per-partner partial attention over the pool (see ``cp_paged_attn_partial`` in cpattn.h)."""
    lib = load_library()
    T, Hq = q.shape[0], q.shape[1]
    B = kv_len.numel() if num_rows is None else num_rows
    st = lib.cp_paged_attn_partial(ctypes.byref(desc), _ptr(pool_k), _ptr(pool_v), _ptr(q), Hq, B, T,
                                   _i32_tensor(qo_indptr, "qo_indptr"), _i32_tensor(kv_len, "kv_len"),
                                   int(max_kv_len), _i32_tensor(kv_page_indptr, "kv_page_indptr"),
                                   _i32_tensor(kv_page_indices, "kv_page_indices"), float(scale), _ptr(o_part),
                                   _ptr(lse_part), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _i32_tensor(dev_status, "dev_status"), _stream(stream))
    _check(st, "cp_paged_attn_partial")


def fused_workspace_bytes(desc: PoolDesc, num_q_heads: int, num_tokens: int, max_kv_len: int) -> int:
    return load_library().cp_paged_attn_fused_workspace_bytes(ctypes.byref(desc), num_q_heads, num_tokens,
                                                              max_kv_len)


def cp_paged_attn_fused(desc: PoolDesc, pool_k, pool_v, q, kv_len, max_kv_len, kv_page_indptr, kv_page_indices,
                        scale, out, workspace, lse_out=None, extra_o=None, extra_lse=None, qo_indptr=None,
                        num_rows=None, row_order=None, dev_status=None, stream=None):
    """All partners' partials and their merge in one launch (see ``cp_paged_attn_fused`` in cpattn.h)."""
    lib = load_library()
    T, Hq = q.shape[0], q.shape[1]
    B = kv_len.numel() if num_rows is None else num_rows
    dt = DTYPE_BF16 if out.dtype == torch.bfloat16 else DTYPE_FP32
    st = lib.cp_paged_attn_fused(ctypes.byref(desc), _ptr(pool_k), _ptr(pool_v), _ptr(q), Hq, B, T,
                                 _i32_tensor(qo_indptr, "qo_indptr"), _i32_tensor(kv_len, "kv_len"),
                                 int(max_kv_len), _i32_tensor(kv_page_indptr, "kv_page_indptr"),
                                 _i32_tensor(kv_page_indices, "kv_page_indices"),
                                 _i32_tensor(row_order, "row_order"), float(scale), _ptr(extra_o),
                                 _ptr(extra_lse), dt, _ptr(out), _ptr(lse_out), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(),
                                 _i32_tensor(dev_status, "dev_status"), _stream(stream))
    _check(st, "cp_paged_attn_fused")


def cp_paged_attn_partial_ex(desc: PoolDesc, pool_k, pool_v, q, kv_len, max_kv_len, kv_page_indptr,
                             kv_page_indices, scale, o_part, lse_part, workspace, lse_layout=LSE_TOKEN_MAJOR,
                             qo_indptr=None, num_rows=None, row_order=None, dev_status=None, stream=None):
    """cp_paged_attn_partial with the LSE layout chosen (see ``cp_paged_attn_partial_ex`` in cpattn.h)."""
    lib = load_library()
    T, Hq = q.shape[0], q.shape[1]
    B = kv_len.numel() if num_rows is None else num_rows
    st = lib.cp_paged_attn_partial_ex(ctypes.byref(desc), _ptr(pool_k), _ptr(pool_v), _ptr(q), Hq, B, T,
                                      _i32_tensor(qo_indptr, "qo_indptr"), _i32_tensor(kv_len, "kv_len"),
                                      int(max_kv_len), _i32_tensor(kv_page_indptr, "kv_page_indptr"),
                                      _i32_tensor(kv_page_indices, "kv_page_indices"), float(scale), _ptr(o_part),
                                      _ptr(lse_part), int(lse_layout), _i32_tensor(row_order, "row_order"),
                                      _ptr(workspace),
                                      workspace.numel() * workspace.element_size(),
                                      _i32_tensor(dev_status, "dev_status"), _stream(stream))
    _check(st, "cp_paged_attn_partial_ex")


def view(o, lse, o_stride_token, o_stride_head, lse_stride_token, lse_stride_head, o_offset=0, lse_offset=0):
    """A cpattn_partial_view of fp32 device tensors (offsets and strides in elements)."""
    if o.dtype != torch.float32 or lse.dtype != torch.float32:
        raise TypeError("partial views are fp32")
    return PartialView(_ptr(o) + 4 * o_offset, _ptr(lse) + 4 * lse_offset, o_stride_token, o_stride_head,
                       lse_stride_token, lse_stride_head)


def lse_merge_views(views, num_tokens, num_heads, head_dim_v, out, out_stride_token, out_stride_head,
                    lse_out=None, lse_out_stride_token=0, lse_out_stride_head=0, out_offset=0, lse_out_offset=0,
                    stream=None):
    """Exact merge of strided partial views (see ``lse_merge_views`` in cpattn.h)."""
    lib = load_library()
    arr = (PartialView * len(views))(*views)
    dt = DTYPE_BF16 if out.dtype == torch.bfloat16 else DTYPE_FP32
    lse_ptr = None if lse_out is None else _ptr(lse_out) + 4 * lse_out_offset
    st = lib.lse_merge_views(len(views), arr, num_tokens, num_heads, head_dim_v, dt,
                             _ptr(out) + out.element_size() * out_offset, out_stride_token, out_stride_head,
                             lse_ptr, lse_out_stride_token, lse_out_stride_head, _stream(stream))
    _check(st, "lse_merge_views")


def own_token_attn(q, k_new, v_new, qo_indptr, num_real_rows, max_q_len, scale, o_own, lse_own, stream=None):
    """Causal attention of the step's new tokens (see ``own_token_attn`` in cpattn.h);
    with ``v_new`` None the value width is ``o_own``'s (MLA: the first 512 key values)."""
    lib = load_library()
    T, Hq, D = q.shape
    Hkv = k_new.shape[1]
    Dv = o_own.shape[-1] if v_new is None else v_new.shape[2]
    dt = DTYPE_BF16 if q.dtype == torch.bfloat16 else DTYPE_FP32
    st = lib.own_token_attn(_ptr(q), _ptr(k_new), _ptr(v_new), Hq, Hkv, D, Dv, dt,
                            _i32_tensor(qo_indptr, "qo_indptr"), qo_indptr.numel() - 1, int(num_real_rows), T,
                            int(max_q_len), float(scale), _ptr(o_own), _ptr(lse_own), _stream(stream))
    _check(st, "own_token_attn")


def lse_merge(o_parts, lse_parts, out, lse_out=None, stream=None):
    """Exact merge of partials ``o_parts [N, T, H, Dv]`` / ``lse_parts [N, T, H]`` into ``out``."""
    lib = load_library()
    N, T, H, Dv = o_parts.shape
    dt = DTYPE_BF16 if out.dtype == torch.bfloat16 else DTYPE_FP32
    st = lib.lse_merge(N, _ptr(o_parts), _ptr(lse_parts), T * H * Dv, T * H, T, H, Dv, dt, _ptr(out),
                       _ptr(lse_out), _stream(stream))
    _check(st, "lse_merge")
