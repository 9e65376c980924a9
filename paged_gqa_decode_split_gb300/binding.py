"""ctypes binding of libpa (include/pa.h): the same entry points under the same
names, with argument marshalling only.  Tensors are passed as raw pointers
(``tensor.data_ptr()``) and streams as ``cudaStream_t`` handles; every step of
the computation runs in libpa's kernels.  There is no fallback: if libpa.so is
missing, every call raises."""
from __future__ import annotations

import ctypes
import os
import re

from . import build as _build

PA_OK = 0
PA_ERR_NULL = -1
PA_ERR_SHAPE = -2
PA_ERR_UNSUPPORTED = -3
PA_ERR_ALIGN = -4
PA_ERR_WORKSPACE = -5
PA_ERR_CUDA = -6
PA_FLAG_BAD_PAGE = 0x1
PA_FLAG_BAD_LENGTH = 0x2
PA_FLAG_TIMEOUT = 0x4
PA_NOALLOC_SCRATCH_BYTES = 16 << 20


class pa_caps(ctypes.Structure):
    _fields_ = [("abi_version", ctypes.c_int32), ("max_batch", ctypes.c_int32), ("max_q_len", ctypes.c_int32),
                ("max_group", ctypes.c_int32), ("page_multiple", ctypes.c_int32), ("max_ctx", ctypes.c_int32),
                ("accum_bits", ctypes.c_int32), ("fp8_head_dim", ctypes.c_int32), ("bf16_head_dim", ctypes.c_int32),
                ("max_splits", ctypes.c_int32), ("reserved", ctypes.c_int32 * 6)]


class pa_params(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("q_len", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("max_pages_per_req", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("max_ctx_len", ctypes.c_int32), ("reserved0", ctypes.c_int32),
                ("k_page_stride", ctypes.c_int64), ("k_token_stride", ctypes.c_int64),
                ("k_head_stride", ctypes.c_int64), ("v_page_stride", ctypes.c_int64),
                ("v_token_stride", ctypes.c_int64), ("v_head_stride", ctypes.c_int64)]


class pa_prefill_params(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("q_len", ctypes.c_int32), ("kv_len", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("k_batch_stride", ctypes.c_int64), ("k_token_stride", ctypes.c_int64),
                ("k_head_stride", ctypes.c_int64), ("v_batch_stride", ctypes.c_int64),
                ("v_token_stride", ctypes.c_int64), ("v_head_stride", ctypes.c_int64)]


_LIB = None
_P = ctypes.POINTER

# pa_bank_alloc_fn / pa_bank_free_fn
BANK_ALLOC_FN = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_void_p)
BANK_FREE_FN = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_void_p)


def lib_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libpa.so (build it first with paged_gqa_decode_split_gb300.build.build())."""
    global _LIB
    if _LIB is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libpa.so not found at {path}: the CUDA library must be built "
                               "(paged_gqa_decode_split_gb300.build.build()); there is no fallback")
        L = ctypes.CDLL(path)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        pp = _P(pa_params)
        sig = {
            "pa_get_capabilities": ([_P(pa_caps)], ctypes.c_int),
            "pa_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "pa_split_plan": ([i32, i32, _P(i32), _P(i32)], ctypes.c_int),
            "pa_decode_fp8_workspace_bytes": ([pp], sz),
            "pa_decode_fp8": ([pp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], ctypes.c_int),
            "pa_decode_fp8_noalloc": ([pp, vp, vp, vp, vp, vp, vp, vp, vp, vp], ctypes.c_int),
            "pa_decode_e5m2": ([pp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], ctypes.c_int),
            "pa_decode_bf16_d128_workspace_bytes": ([pp], sz),
            "pa_decode_bf16_d128": ([pp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], ctypes.c_int),
            "pa_decode_bf16_d256": ([pp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], ctypes.c_int),
            "pa_decode_f16": ([pp, vp, vp, vp, vp, vp, vp, vp, sz, vp], ctypes.c_int),
            "pa_prefill_plan": ([i32, _P(i32), _P(i32)], ctypes.c_int),
            "pa_prefill_f16_workspace_bytes": ([_P(pa_prefill_params)], sz),
            "pa_prefill_f16": ([_P(pa_prefill_params), vp, vp, vp, vp, vp, vp, sz, vp], ctypes.c_int),
            "pa_bank_create": ([BANK_ALLOC_FN, BANK_FREE_FN, vp], vp),
            "pa_bank_destroy": ([vp], ctypes.c_int),
            "pa_bank_workspace": ([vp, pp, i32, vp, _P(vp), _P(sz)], ctypes.c_int),
            "pa_bank_stats": ([vp, _P(i64), _P(i64)], ctypes.c_int),
            "pa_read_status": ([vp, _P(ctypes.c_uint32), vp], ctypes.c_int),
            "pa_clear_status": ([vp, vp], ctypes.c_int),
            "pa_debug_worklist": ([pp, vp, vp, i32, vp, vp], ctypes.c_int),
            "pa_debug_gather_fp8": ([pp, vp, vp, vp, vp, i32, vp, vp], ctypes.c_int),
            "pa_debug_kv_load_path": ([pp, i32, i32, vp, vp, _P(i32)], ctypes.c_int),
            "pa_debug_stall_next": ([i64], ctypes.c_int),
            "pa_timing_enable": ([ctypes.c_int], ctypes.c_int),
            "pa_timing_collect": ([ctypes.c_int, _P(ctypes.c_double), _P(i64)], ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _LIB = L
    return _LIB


def header_functions() -> list[str]:
    """Names of the functions declared in include/pa.h."""
    text = open(os.path.join(_build.INCLUDE, "pa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


# ---------------------------------------------------------------- marshalling --

def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def status_string(status: int) -> str:
    return load().pa_status_string(int(status)).decode()


def check(status: int, what: str = "libpa call") -> None:
    if status != PA_OK:
        raise RuntimeError(f"{what} failed: {status} ({status_string(status)})")


def make_params(*, batch, num_kv_heads, num_q_heads, head_dim, q_len, page_size, max_pages_per_req, num_pages,
                max_ctx_len, k_strides, v_strides) -> pa_params:
    p = pa_params()
    p.batch, p.num_kv_heads, p.num_q_heads, p.head_dim = batch, num_kv_heads, num_q_heads, head_dim
    p.q_len, p.page_size, p.max_pages_per_req, p.num_pages = q_len, page_size, max_pages_per_req, num_pages
    p.max_ctx_len = max_ctx_len
    p.k_page_stride, p.k_token_stride, p.k_head_stride = (int(s) for s in k_strides)
    p.v_page_stride, p.v_token_stride, p.v_head_stride = (int(s) for s in v_strides)
    return p


def pa_get_capabilities() -> pa_caps:
    c = pa_caps()
    check(load().pa_get_capabilities(ctypes.byref(c)), "pa_get_capabilities")
    return c


def pa_split_plan(ctx_len: int, num_kv_heads: int = 1) -> tuple[int, int, int]:
    s, c = ctypes.c_int32(), ctypes.c_int32()
    st = load().pa_split_plan(int(ctx_len), int(num_kv_heads), ctypes.byref(s), ctypes.byref(c))
    return st, s.value, c.value


def pa_prefill_plan(kv_len: int) -> tuple[int, int, int]:
    """(status, num_splits, split_len) of the prefill key split."""
    s, c = ctypes.c_int32(), ctypes.c_int32()
    st = load().pa_prefill_plan(int(kv_len), ctypes.byref(s), ctypes.byref(c))
    return st, s.value, c.value


def pa_prefill_f16_workspace_bytes(p: pa_prefill_params) -> int:
    return int(load().pa_prefill_f16_workspace_bytes(ctypes.byref(p)))


def pa_prefill_f16(p: pa_prefill_params, q, k, v, out, lse, workspace, workspace_bytes: int, stream=None) -> int:
    return load().pa_prefill_f16(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(workspace),
                                 int(workspace_bytes), _stream(stream))


def pa_decode_fp8_workspace_bytes(p: pa_params) -> int:
    return int(load().pa_decode_fp8_workspace_bytes(ctypes.byref(p)))


def pa_decode_bf16_d128_workspace_bytes(p: pa_params) -> int:
    return int(load().pa_decode_bf16_d128_workspace_bytes(ctypes.byref(p)))


def pa_decode_fp8(p: pa_params, q, k_pages, v_pages, block_table, ctx_lens, k_scale, v_scale, out, workspace,
                  workspace_bytes: int, stream=None) -> int:
    return load().pa_decode_fp8(ctypes.byref(p), _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                _ptr(ctx_lens), _ptr(k_scale), _ptr(v_scale), _ptr(out), _ptr(workspace),
                                int(workspace_bytes), _stream(stream))


def pa_decode_e5m2(p: pa_params, q, k_pages, v_pages, block_table, ctx_lens, k_scale, v_scale, out, workspace,
                   workspace_bytes: int, stream=None) -> int:
    return load().pa_decode_e5m2(ctypes.byref(p), _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                 _ptr(ctx_lens), _ptr(k_scale), _ptr(v_scale), _ptr(out), _ptr(workspace),
                                 int(workspace_bytes), _stream(stream))


def pa_decode_fp8_noalloc(p: pa_params, q, k_pages, v_pages, block_table, ctx_lens, k_scale, v_scale, out,
                          stream=None) -> int:
    return load().pa_decode_fp8_noalloc(ctypes.byref(p), _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                        _ptr(ctx_lens), _ptr(k_scale), _ptr(v_scale), _ptr(out), _stream(stream))


def pa_decode_bf16_d128(p: pa_params, q, k_pages, v_pages, block_table, ctx_lens, out, lse, workspace,
                        workspace_bytes: int, stream=None) -> int:
    return load().pa_decode_bf16_d128(ctypes.byref(p), _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                      _ptr(ctx_lens), _ptr(out), _ptr(lse), _ptr(workspace), int(workspace_bytes),
                                      _stream(stream))


def pa_bank_create(alloc_fn, free_fn=None):
    """alloc_fn(nbytes, device) -> device address (int, zero-filled, 256-byte
    aligned) or 0; free_fn(ptr, nbytes, device) or None.  Returns (handle,
    keepalive): keep `keepalive` referenced for as long as the bank lives."""
    a = BANK_ALLOC_FN(lambda n, dev, user: alloc_fn(int(n), int(dev)) or None)
    f = BANK_FREE_FN(lambda ptr, n, dev, user: free_fn(int(ptr or 0), int(n), int(dev))) if free_fn else \
        ctypes.cast(None, BANK_FREE_FN)
    h = load().pa_bank_create(a, f, None)
    return h, (a, f)


def pa_bank_destroy(bank) -> int:
    return load().pa_bank_destroy(bank)


def pa_bank_workspace(bank, p: pa_params, device: int, stream) -> tuple[int, int, int]:
    """Returns (status, workspace address, workspace bytes).  `stream` is only
    a key: an int (cudaStream_t), a torch stream or None (the legacy default
    stream, 0)."""
    ws, n = ctypes.c_void_p(), ctypes.c_size_t()
    key = 0 if stream is None else (stream if isinstance(stream, int) else stream.cuda_stream)
    st = load().pa_bank_workspace(bank, ctypes.byref(p), int(device), key, ctypes.byref(ws), ctypes.byref(n))
    return st, int(ws.value or 0), int(n.value)


def pa_bank_stats(bank) -> tuple[int, int, int]:
    panels, nbytes = ctypes.c_int64(), ctypes.c_int64()
    st = load().pa_bank_stats(bank, ctypes.byref(panels), ctypes.byref(nbytes))
    return st, panels.value, nbytes.value


def pa_decode_f16(p: pa_params, q, k_pages, v_pages, block_table, ctx_lens, out, workspace, workspace_bytes: int,
                  stream=None) -> int:
    return load().pa_decode_f16(ctypes.byref(p), _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                _ptr(ctx_lens), _ptr(out), _ptr(workspace), int(workspace_bytes), _stream(stream))


def pa_decode_bf16_d256(p: pa_params, q, k_pages, v_pages, block_table, ctx_lens, out, lse, workspace,
                        workspace_bytes: int, stream=None) -> int:
    return load().pa_decode_bf16_d256(ctypes.byref(p), _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                      _ptr(ctx_lens), _ptr(out), _ptr(lse), _ptr(workspace), int(workspace_bytes),
                                      _stream(stream))


def pa_read_status(workspace, stream=None) -> tuple[int, int]:
    f = ctypes.c_uint32()
    st = load().pa_read_status(_ptr(workspace), ctypes.byref(f), _stream(stream))
    return st, f.value


def pa_clear_status(workspace, stream=None) -> int:
    return load().pa_clear_status(_ptr(workspace), _stream(stream))


def pa_debug_worklist(p: pa_params, ctx_lens, items, max_items: int, count, stream=None) -> int:
    return load().pa_debug_worklist(ctypes.byref(p), _ptr(ctx_lens), _ptr(items), int(max_items), _ptr(count),
                                    _stream(stream))


def pa_debug_gather_fp8(p: pa_params, k_pages, v_pages, block_table, ctx_lens, which: int, dst, stream=None) -> int:
    return load().pa_debug_gather_fp8(ctypes.byref(p), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                      _ptr(ctx_lens), int(which), _ptr(dst), _stream(stream))


PA_KV_LOAD_COPY, PA_KV_LOAD_TMA, PA_KV_LOAD_WINDOW = 0, 1, 2


def pa_debug_kv_load_path(p: pa_params, head_dim: int, elem_bytes: int, k_pages, v_pages) -> tuple[int, int]:
    """(status, path): how a decode call with this geometry and these K/V
    bases loads K and V (PA_KV_LOAD_*)."""
    path = ctypes.c_int32(-1)
    st = load().pa_debug_kv_load_path(ctypes.byref(p), int(head_dim), int(elem_bytes), _ptr(k_pages),
                                      _ptr(v_pages), ctypes.byref(path))
    return st, path.value


def pa_debug_stall_next(wait_limit_cycles: int) -> int:
    return load().pa_debug_stall_next(int(wait_limit_cycles))


def pa_timing_enable(on: bool) -> int:
    return load().pa_timing_enable(1 if on else 0)


def pa_timing_collect(kernel: int) -> tuple[int, float, int]:
    ms, n = ctypes.c_double(), ctypes.c_int64()
    st = load().pa_timing_collect(int(kernel), ctypes.byref(ms), ctypes.byref(n))
    return st, ms.value, n.value
