"""FP64 CPU oracle for paged GQA decode / speculative-verify attention.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package.  It shares no code with ``paged_gqa_decode_split_gb300`` and does
not import it; both sides only consume the same seeded inputs.

The arithmetic lives in ``paged_attn_oracle.c`` (plain C, double precision,
OpenMP over output rows), which is compiled on first use with the host C
compiler.  This module only marshals numpy arrays into that library.

Sources followed (see the C file for the full statement of the definition):
  * "DFlash2 concurrent long-context attention", sections "Why the
    single-request optimization was missing from concurrent decode" (E4M3 KV,
    FP16 Q, D = 256, GQA 6, multiple six-head groups, zero-length and padded
    rows safe) and "Operator validation" (independent FP64 oracle).
  * "SM70 attention and quantized projection coverage across TP sizes",
    section "Scope" (FP32 or better accumulation for QK and PV).
  * "perf(fa2): port decode GQA group-swap into d128 varlen launcher" (vllm.cpp
    pull request #48), description: the BF16 head-dim-128 decode variant.
  * E5M2 K/V, a cache type the first page names beside E4M3 (same section as
    above) and whose graphs "SM70 attention and quantized projection coverage
    across TP sizes", section "Additional findings", checks against FP64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "paged_attn_oracle.c")
_LOCK = threading.Lock()
_LIBS: dict[int, ctypes.CDLL] = {}


def build(mutation: int = 0, out_dir: str | None = None) -> str:
    """Compile the oracle with gcc (OpenMP) and return the path of the .so.

    ``mutation`` != 0 plants the numbered deliberate mistake (pin-strength
    tests only); such builds go to ``out_dir``.
    """
    out_dir = out_dir or os.path.join(_HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    name = "liboracle.so" if mutation == 0 else f"liboracle_mut{mutation}.so"
    path = os.path.join(out_dir, name)
    if os.path.exists(path) and os.path.getmtime(path) >= os.path.getmtime(_SRC):
        return path
    tmp = path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC", f"-DORACLE_MUTATION={mutation}",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)
    return path


def _setup(lib: ctypes.CDLL) -> ctypes.CDLL:
    i32, i64, f32, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
    lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_value.restype = ctypes.c_double
    lib.oracle_e5m2_value.argtypes = [ctypes.c_uint8]
    lib.oracle_e5m2_value.restype = ctypes.c_double
    lib.oracle_f16_value.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_value.restype = ctypes.c_double
    lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_value.restype = ctypes.c_double
    common = [i32] * 7 + [vp, vp, vp] + [i64] * 6 + [vp, vp]
    lib.oracle_paged_attn_fp8.argtypes = common + [f32, f32, vp, i32, vp, vp, i32]
    lib.oracle_paged_attn_fp8.restype = i32
    lib.oracle_paged_attn_e5m2.argtypes = common + [f32, f32, vp, i32, vp, vp, i32]
    lib.oracle_paged_attn_e5m2.restype = i32
    lib.oracle_paged_attn_bf16.argtypes = common + [vp, i32, vp, vp, i32]
    lib.oracle_paged_attn_f16.argtypes = common + [vp, i32, vp, vp, i32]
    lib.oracle_paged_attn_f16.restype = i32
    lib.oracle_paged_attn_bf16.restype = i32
    lib.oracle_max_threads.restype = i32
    lib.oracle_mutation.restype = i32
    return lib


def load(mutation: int = 0, out_dir: str | None = None) -> ctypes.CDLL:
    with _LOCK:
        key = mutation if out_dir is None else hash((mutation, out_dir))
        if key not in _LIBS:
            _LIBS[key] = _setup(ctypes.CDLL(build(mutation, out_dir)))
        return _LIBS[key]


def max_threads(lib: ctypes.CDLL | None = None) -> int:
    return int((lib or load()).oracle_max_threads())


def e4m3_value(codes, lib=None) -> np.ndarray:
    lib = lib or load()
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.oracle_e4m3_value(int(x)) for x in c], dtype=np.float64)


def e5m2_value(codes, lib=None) -> np.ndarray:
    lib = lib or load()
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.oracle_e5m2_value(int(x)) for x in c], dtype=np.float64)


def f16_value(bits, lib=None) -> np.ndarray:
    lib = lib or load()
    c = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.oracle_f16_value(int(x)) for x in c], dtype=np.float64)


def bf16_value(bits, lib=None) -> np.ndarray:
    lib = lib or load()
    c = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.oracle_bf16_value(int(x)) for x in c], dtype=np.float64)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def paged_attn(kind: str, *, q: np.ndarray, kv: np.ndarray, k_offset: int, v_offset: int,
               k_strides: tuple[int, int, int], v_strides: tuple[int, int, int],
               block_table: np.ndarray, ctx_lens: np.ndarray, num_kv_heads: int, page_size: int,
               k_scale: float = 1.0, v_scale: float = 1.0, rows=None, num_threads: int = 0, lib=None):
    """Evaluate the definition for every (or the selected) output rows.

    kind          "fp8" (FP16 Q, E4M3 K/V + FP32 scales), "e5m2" (FP16 Q, E5M2
                  K/V + FP32 scales), "f16" (FP16 Q/K/V) or "bf16" (BF16 Q/K/V).
    q             uint16 bit patterns [B, q_len, Hq, D].
    kv            one uint8 host buffer holding both K and V pages; K element
                  (page, slot, head, d) is at byte k_offset + page*k_strides[0]
                  + slot*k_strides[1] + head*k_strides[2] + d*elem_size, and V
                  likewise with v_offset / v_strides.
    block_table   int32 [B, max_pages_per_req]; ctx_lens int32 [B].
    rows          None for all rows, else flat row ids (b*q_len + qi)*Hq + h.
    Returns (out float64 [..., D], lse float64 [...]).
    """
    lib = lib or load()
    q = np.ascontiguousarray(q).view(np.uint16)
    B, q_len, Hq, D = q.shape
    kv = np.ascontiguousarray(kv).view(np.uint8)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    cl = np.ascontiguousarray(ctx_lens, dtype=np.int32)
    if rows is None:
        out = np.empty((B, q_len, Hq, D), np.float64)
        lse = np.empty((B, q_len, Hq), np.float64)
        rows_arr, n_rows, rows_ptr = None, 0, None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int32)
        n_rows = int(rows_arr.size)
        out = np.empty((n_rows, D), np.float64)
        lse = np.empty((n_rows,), np.float64)
        rows_ptr = _ptr(rows_arr)
    base = _ptr(kv)
    args = [B, q_len, Hq, num_kv_heads, D, page_size, bt.shape[1], _ptr(q), base + k_offset, base + v_offset,
            *[int(s) for s in k_strides], *[int(s) for s in v_strides], _ptr(bt), _ptr(cl)]
    if kind in ("fp8", "e5m2"):
        fn = lib.oracle_paged_attn_fp8 if kind == "fp8" else lib.oracle_paged_attn_e5m2
        rc = fn(*args, float(k_scale), float(v_scale), rows_ptr, n_rows, _ptr(out), _ptr(lse), int(num_threads))
    elif kind in ("bf16", "f16"):
        fn = lib.oracle_paged_attn_bf16 if kind == "bf16" else lib.oracle_paged_attn_f16
        rc = fn(*args, rows_ptr, n_rows, _ptr(out), _ptr(lse), int(num_threads))
    else:
        raise ValueError(kind)
    if rc != 0:
        raise RuntimeError(f"oracle failed with status {rc}")
    return out, lse


def prefill_attn(*, q: np.ndarray, k: np.ndarray, v: np.ndarray, k_strides: tuple[int, int, int],
                 v_strides: tuple[int, int, int], kv_len: int, num_kv_heads: int, rows=None, num_threads: int = 0,
                 lib=None):
    """The causal long prefill ("SM70 attention and quantized projection
    coverage across TP sizes", sections "Scope" and "Accumulation audit and
    rejected tuning": Q8192 x KV262144, FP16 inputs) is the same definition
    with q_len prefill queries that are the last q_len positions of a
    kv_len-key context: query i sees keys 0 .. kv_len - q_len + i.  A request's
    dense K and V are one page of kv_len slots, page b for request b.

    q        uint16 FP16 bits [B, q_len, Hq, D].
    k, v     uint16 FP16 bits, flat buffers; element (b, key t, kv head g, d)
             of K at k[b*k_strides[0] + t*k_strides[1] + g*k_strides[2] + d]
             (element strides), V likewise.
    rows     None for all rows, else flat row ids (b*q_len + i)*Hq + h.
    Returns (out float64, lse float64) as ``paged_attn``.
    """
    lib = lib or load()
    q = np.ascontiguousarray(q).view(np.uint16)
    B, q_len, Hq, D = q.shape
    k = np.ascontiguousarray(k).view(np.uint16)
    v = np.ascontiguousarray(v).view(np.uint16)
    bt = np.arange(B, dtype=np.int32).reshape(B, 1)
    cl = np.full(B, int(kv_len), dtype=np.int32)
    if rows is None:
        out = np.empty((B, q_len, Hq, D), np.float64)
        lse = np.empty((B, q_len, Hq), np.float64)
        rows_arr, n_rows, rows_ptr = None, 0, None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int32)
        n_rows = int(rows_arr.size)
        out = np.empty((n_rows, D), np.float64)
        lse = np.empty((n_rows,), np.float64)
        rows_ptr = _ptr(rows_arr)
    rc = lib.oracle_paged_attn_f16(B, q_len, Hq, num_kv_heads, D, int(kv_len), 1, _ptr(q), _ptr(k), _ptr(v),
                                   *[2 * int(s) for s in k_strides], *[2 * int(s) for s in v_strides], _ptr(bt),
                                   _ptr(cl), rows_ptr, n_rows, _ptr(out), _ptr(lse), int(num_threads))
    if rc != 0:
        raise RuntimeError(f"oracle failed with status {rc}")
    return out, lse
