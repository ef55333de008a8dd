"""Python binding of libpagedattn: attention over a paged KV cache on GB300.

Argument marshalling only.  Each ``pa_*`` function here has the name and
argument order of the C entry point in ``include/pagedattn.h``; tensors stand
in for device pointers (``None`` for a NULL pointer) and ``stream`` defaults to
PyTorch's current stream.  Every step of the computation runs in the
library's CUDA kernels; if the library is missing, loading it raises -- there
is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "lib", "libpagedattn.so")

PA_OK = 0
PA_ERR_NULL = 1
PA_ERR_DTYPE = 2
PA_ERR_SHAPE = 3
PA_ERR_ALIGN = 4
PA_ERR_UNSUPPORTED = 5
PA_ERR_WORKSPACE = 6
PA_ERR_CUDA = 7
PA_ERR_VALIDATION = 8
PA_ERR_CAPACITY = 9

PA_F32 = 0
PA_BF16 = 1

PA_DEVERR_BAD_SLOT = 0x1
PA_DEVERR_BAD_PAGE = 0x2
PA_DEVERR_BAD_LENGTH = 0x4
PA_DEVERR_TIMEOUT = 0x8


class PagedAttnError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        extra = f" (cudaError {cuda_error})" if status == PA_ERR_CUDA else ""
        super().__init__(f"{fn}: status {status}: {message}{extra}")


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_pages", ctypes.c_int64), ("dtype", ctypes.c_int32)]


def cache_desc(num_q_heads: int, num_kv_heads: int, head_dim: int, page_size: int, num_pages: int,
               dtype) -> CacheDesc:
    """Build a descriptor; ``dtype`` is torch.float32 / torch.bfloat16 or PA_F32 / PA_BF16."""
    if dtype in (torch.float32, PA_F32):
        code = PA_F32
    elif dtype in (torch.bfloat16, PA_BF16):
        code = PA_BF16
    else:
        code = int(dtype) if isinstance(dtype, int) else -1
    return CacheDesc(num_q_heads, num_kv_heads, head_dim, page_size, num_pages, code)


_lib: Optional[ctypes.CDLL] = None

_VP = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_F32 = ctypes.c_float
_DESC = ctypes.POINTER(CacheDesc)

_SIGS = {
    "pa_slot_mapping": (_I32, [_DESC, _I32, _VP, _VP, _VP, _I32, _I64, _VP, _VP, _VP]),
    "pa_kv_write": (_I32, [_DESC, _VP, _I64, _VP, _I64, _I64, _VP, _VP, _VP, _VP]),
    "pa_qk_norm_rope_kv_write": (_I32, [_DESC, _VP, _I64, _VP, _I64, _VP, _I64, _I64, _VP, _VP, _VP, _F32, _F32,
                                        _VP, _VP, _VP, _VP, _VP]),
    "pa_prefill_qk_norm_rope_kv_write": (_I32, [_DESC, _VP, _I64, _VP, _I64, _VP, _I64, _I64, _VP, _I32, _VP, _VP,
                                                _I32, _VP, _VP, _F32, _F32, _VP, _VP, _VP, _VP, _VP, _VP]),
    "pa_decode_workspace_size": (ctypes.c_size_t, [_DESC, _I32, _I32, _I32]),
    "pa_decode_plan_info": (_I32, [_DESC, _I32, _I32, _I32, ctypes.POINTER(_I32), ctypes.POINTER(_I32)]),
    "pa_decode": (_I32, [_DESC, _VP, _I32, _VP, _VP, _VP, _I32, _VP, _I32, _F32, _I32, _VP, _VP, ctypes.c_size_t,
                         _VP]),
    "pa_decode_kv_write": (_I32, [_DESC, _VP, _VP, _I64, _VP, _I64, _I32, _VP, _VP, _VP, _I32, _VP, _I32, _F32, _I32,
                                  _VP, _VP, _VP, ctypes.c_size_t, _VP]),
    "pa_decode_no_alloc": (_I32, [_DESC, _VP, _I32, _VP, _VP, _VP, _I32, _VP, _I32, _F32, _I32, _VP, _VP]),
    "pa_prefill_varlen": (_I32, [_DESC, _VP, _VP, _I32, _I32, _I64, _VP, _VP, _VP, _I32, _VP, _I32, _F32, _VP, _VP,
                                 ctypes.c_size_t, _VP]),
    "pa_prefill_step": (_I32, [_DESC, _VP, _I64, _VP, _I64, _VP, _I64, _I64, _VP, _I32, _I32, _VP, _I32, _VP, _I32,
                               _VP, _VP, _F32, _F32, _F32, _VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_size_t, _VP]),
    "pa_prefill_workspace_size": (ctypes.c_size_t, [_DESC, _I32, _I32, _I64, _I32]),
    "pa_validate_metadata": (_I32, [_DESC, _I32, _VP, _VP, _VP, _I32, _I32, _VP, _VP]),
    "pa_selftest_bounded_wait": (_I32, [_I32, _VP]),
    "pa_read_device_errors": (_I32, [ctypes.POINTER(ctypes.c_uint32), _I32]),
    "pa_last_cuda_error": (_I32, []),
    "pa_status_string": (ctypes.c_char_p, [_I32]),
    "pa_version": (_I32, []),
    "pa_bm_create": (_I32, [_I64, _I32, ctypes.POINTER(_VP)]),
    "pa_bm_destroy": (None, [_VP]),
    "pa_bm_can_allocate": (_I32, [_VP, _VP, _I64, ctypes.POINTER(_I64)]),
    "pa_bm_allocate": (_I32, [_VP, _I64, _VP, _I64, ctypes.POINTER(_I64)]),
    "pa_bm_append_token": (_I32, [_VP, _I64, _I32]),
    "pa_bm_hash_blocks": (_I32, [_VP, _I64, _I64]),
    "pa_bm_free": (_I32, [_VP, _I64]),
    "pa_bm_block_tables": (_I32, [_VP, _VP, _I32, _I32, _I32, _VP, _VP]),
    "pa_bm_slot_mapping": (_I32, [_VP, _VP, _I32, _VP, _VP]),
    "pa_bm_query": (_I32, [_VP, ctypes.POINTER(_I64), ctypes.POINTER(_I64), ctypes.POINTER(_I64)]),
    "pa_bm_block_ref_count": (_I32, [_VP, _I32, ctypes.POINTER(_I32)]),
    "pa_bm_seq_info": (_I32, [_VP, _I64, ctypes.POINTER(_I64), ctypes.POINTER(_I64), ctypes.POINTER(_I32)]),
}


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libpagedattn.so (built by ``paged_kv_gqa_08_gb300.build``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"libpagedattn.so not found at {p}; build it with "
                          "`python -m paged_kv_gqa_08_gb300.build`")
    lib = ctypes.CDLL(p)
    for name, (res, args) in _SIGS.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    if path is None:
        _lib = lib
    return lib


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return t.data_ptr() if t.numel() > 0 else None
    return int(t)


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(fn: str, status: int) -> None:
    if status != PA_OK:
        lib = load_library()
        msg = lib.pa_status_string(status).decode()
        raise PagedAttnError(fn, status, msg, lib.pa_last_cuda_error())


def pa_slot_mapping(desc, batch, cu_seqlens_q, context_lens, block_tables, max_pages_per_seq, num_tokens,
                    positions, slot_mapping, stream=None):
    lib = load_library()
    _check("pa_slot_mapping", lib.pa_slot_mapping(
        ctypes.byref(desc), batch, _ptr(cu_seqlens_q), _ptr(context_lens), _ptr(block_tables),
        max_pages_per_seq, num_tokens, _ptr(positions), _ptr(slot_mapping), _stream(stream)))


def pa_kv_write(desc, k, k_row_stride, v, v_row_stride, num_tokens, slot_mapping, k_cache, v_cache, stream=None):
    lib = load_library()
    _check("pa_kv_write", lib.pa_kv_write(
        ctypes.byref(desc), _ptr(k), k_row_stride, _ptr(v), v_row_stride, num_tokens, _ptr(slot_mapping),
        _ptr(k_cache), _ptr(v_cache), _stream(stream)))


def pa_qk_norm_rope_kv_write(desc, q, q_row_stride, k, k_row_stride, v, v_row_stride, num_tokens, positions,
                             q_norm_w, k_norm_w, eps, rope_theta, slot_mapping, q_out, k_cache, v_cache,
                             stream=None):
    lib = load_library()
    _check("pa_qk_norm_rope_kv_write", lib.pa_qk_norm_rope_kv_write(
        ctypes.byref(desc), _ptr(q), q_row_stride, _ptr(k), k_row_stride, _ptr(v), v_row_stride, num_tokens,
        _ptr(positions), _ptr(q_norm_w), _ptr(k_norm_w), eps, rope_theta, _ptr(slot_mapping), _ptr(q_out),
        _ptr(k_cache), _ptr(v_cache), _stream(stream)))


def pa_prefill_qk_norm_rope_kv_write(desc, q, q_row_stride, k, k_row_stride, v, v_row_stride, num_tokens,
                                     cu_seqlens_q, batch, context_lens, block_tables, max_pages_per_seq, q_norm_w,
                                     k_norm_w, eps, rope_theta, q_out, k_cache, v_cache, positions_out=None,
                                     slot_mapping_out=None, stream=None):
    lib = load_library()
    _check("pa_prefill_qk_norm_rope_kv_write", lib.pa_prefill_qk_norm_rope_kv_write(
        ctypes.byref(desc), _ptr(q), q_row_stride, _ptr(k), k_row_stride, _ptr(v), v_row_stride, num_tokens,
        _ptr(cu_seqlens_q), batch, _ptr(context_lens), _ptr(block_tables), max_pages_per_seq, _ptr(q_norm_w),
        _ptr(k_norm_w), eps, rope_theta, _ptr(q_out), _ptr(k_cache), _ptr(v_cache), _ptr(positions_out),
        _ptr(slot_mapping_out), _stream(stream)))


def pa_decode_workspace_size(desc, batch, max_context_len, max_ctas=0) -> int:
    return int(load_library().pa_decode_workspace_size(ctypes.byref(desc), batch, max_context_len, max_ctas))


def pa_decode_plan_info(desc, batch, max_context_len, max_ctas=0):
    """(num_partitions, tokens_per_chunk) pa_decode would use on the current device."""
    lib = load_library()
    n = _I32(0)
    t = _I32(0)
    _check("pa_decode_plan_info", lib.pa_decode_plan_info(ctypes.byref(desc), batch, max_context_len, max_ctas,
                                                          ctypes.byref(n), ctypes.byref(t)))
    return int(n.value), int(t.value)


def pa_decode(desc, q, batch, k_cache, v_cache, block_tables, max_pages_per_seq, context_lens, max_context_len,
              scale, max_ctas, out, workspace, workspace_bytes=None, stream=None):
    lib = load_library()
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("pa_decode", lib.pa_decode(
        ctypes.byref(desc), _ptr(q), batch, _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), max_pages_per_seq,
        _ptr(context_lens), max_context_len, scale, max_ctas, _ptr(out), _ptr(workspace), workspace_bytes,
        _stream(stream)))


def pa_decode_kv_write(desc, q, k_new, k_row_stride, v_new, v_row_stride, batch, k_cache, v_cache, block_tables,
                       max_pages_per_seq, context_lens, max_context_len, scale, max_ctas, slot_mapping, out, workspace,
                       workspace_bytes=None, stream=None):
    lib = load_library()
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("pa_decode_kv_write", lib.pa_decode_kv_write(
        ctypes.byref(desc), _ptr(q), _ptr(k_new), k_row_stride, _ptr(v_new), v_row_stride, batch, _ptr(k_cache),
        _ptr(v_cache), _ptr(block_tables), max_pages_per_seq, _ptr(context_lens), max_context_len, scale, max_ctas,
        _ptr(slot_mapping), _ptr(out), _ptr(workspace), workspace_bytes, _stream(stream)))


def pa_decode_no_alloc(desc, q, batch, k_cache, v_cache, block_tables, max_pages_per_seq, context_lens,
                       max_context_len, scale, max_ctas, out, stream=None):
    """pa_decode with the library's fixed 16 MiB scratch instead of a caller workspace."""
    lib = load_library()
    _check("pa_decode_no_alloc", lib.pa_decode_no_alloc(
        ctypes.byref(desc), _ptr(q), batch, _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), max_pages_per_seq,
        _ptr(context_lens), max_context_len, scale, max_ctas, _ptr(out), _stream(stream)))


def pa_prefill_varlen(desc, q, cu_seqlens_q, batch, max_seqlen_q, num_tokens, k_cache, v_cache, block_tables,
                      max_pages_per_seq, context_lens, max_context_len, scale, out, workspace=None,
                      workspace_bytes=None, stream=None):
    lib = load_library()
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("pa_prefill_varlen", lib.pa_prefill_varlen(
        ctypes.byref(desc), _ptr(q), _ptr(cu_seqlens_q), batch, max_seqlen_q, num_tokens, _ptr(k_cache),
        _ptr(v_cache), _ptr(block_tables), max_pages_per_seq, _ptr(context_lens), max_context_len, scale,
        _ptr(out), _ptr(workspace), workspace_bytes, _stream(stream)))


def pa_prefill_step(desc, q, q_row_stride, k, k_row_stride, v, v_row_stride, num_tokens, cu_seqlens_q, batch,
                    max_seqlen_q, context_lens, max_context_len, block_tables, max_pages_per_seq, q_norm_w, k_norm_w,
                    eps, rope_theta, scale, q_out, k_cache, v_cache, positions_out, slot_mapping_out, out,
                    workspace=None, workspace_bytes=None, stream=None):
    lib = load_library()
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("pa_prefill_step", lib.pa_prefill_step(
        ctypes.byref(desc), _ptr(q), q_row_stride, _ptr(k), k_row_stride, _ptr(v), v_row_stride, num_tokens,
        _ptr(cu_seqlens_q), batch, max_seqlen_q, _ptr(context_lens), max_context_len, _ptr(block_tables),
        max_pages_per_seq, _ptr(q_norm_w), _ptr(k_norm_w), eps, rope_theta, scale, _ptr(q_out), _ptr(k_cache),
        _ptr(v_cache), _ptr(positions_out), _ptr(slot_mapping_out), _ptr(out), _ptr(workspace), workspace_bytes,
        _stream(stream)))


def pa_prefill_workspace_size(desc, batch, max_seqlen_q, num_tokens, max_context_len) -> int:
    return int(load_library().pa_prefill_workspace_size(ctypes.byref(desc), batch, max_seqlen_q, num_tokens,
                                                        max_context_len))


def pa_validate_metadata(desc, batch, cu_seqlens_q, context_lens, block_tables, max_pages_per_seq,
                         max_context_len, error_count, stream=None):
    lib = load_library()
    _check("pa_validate_metadata", lib.pa_validate_metadata(
        ctypes.byref(desc), batch, _ptr(cu_seqlens_q), _ptr(context_lens), _ptr(block_tables), max_pages_per_seq,
        max_context_len, _ptr(error_count), _stream(stream)))


def pa_selftest_bounded_wait(timeout_ms: int, stream=None):
    _check("pa_selftest_bounded_wait", load_library().pa_selftest_bounded_wait(timeout_ms, _stream(stream)))


def pa_read_device_errors(reset: bool = False) -> int:
    lib = load_library()
    flags = ctypes.c_uint32(0)
    _check("pa_read_device_errors", lib.pa_read_device_errors(ctypes.byref(flags), 1 if reset else 0))
    return int(flags.value)


def pa_status_string(status: int) -> str:
    return load_library().pa_status_string(status).decode()


def pa_version() -> int:
    return int(load_library().pa_version())
