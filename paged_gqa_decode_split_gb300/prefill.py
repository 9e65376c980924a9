"""Convenience call over the C ABI for causal prefill workloads held in torch
tensors (pa_prefill_f16).  Device memory (output, LSE, workspace) is
allocated with torch; the arithmetic runs in libpa's kernels."""
from __future__ import annotations

import torch

from . import binding as B
from .workloads import PrefillWorkload


def prefill_params(w: PrefillWorkload) -> B.pa_prefill_params:
    s = w.spec
    p = B.pa_prefill_params()
    p.batch, p.q_len, p.kv_len = s.batch, s.q_len, s.kv_len
    p.num_q_heads, p.num_kv_heads, p.head_dim = s.num_q_heads, s.num_kv_heads, s.head_dim
    p.k_batch_stride, p.k_token_stride, p.k_head_stride = (int(x) for x in w.k_strides)
    p.v_batch_stride, p.v_token_stride, p.v_head_stride = (int(x) for x in w.v_strides)
    return p


def logical_causal_flops(batch: int, q_len: int, kv_len: int, num_q_heads: int, head_dim: int) -> int:
    """4 * D * Hq * (visible (query, key) pairs): the QK and PV products of
    every key each query sees, two FLOPs per multiply-add."""
    n = min(q_len, kv_len)
    # queries q_len - n .. q_len - 1 see kv_len - n + 1 .. kv_len keys
    pairs = n * (kv_len - n) + n * (n + 1) // 2
    return 4 * head_dim * num_q_heads * batch * pairs


class Prefill:
    """Holds the output, LSE and workspace of one prefill workload and
    enqueues pa_prefill_f16 on a stream."""

    def __init__(self, w: PrefillWorkload, *, with_lse: bool = True):
        if not w.q.is_cuda:
            raise ValueError("the workload must be on a CUDA device")
        self.w = w
        self.p = prefill_params(w)
        self.ws_bytes = B.pa_prefill_f16_workspace_bytes(self.p)
        if self.ws_bytes == 0:
            raise ValueError("libpa rejects this prefill geometry")
        dev = w.q.device
        self.workspace = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.out = torch.empty_like(w.q)
        self.lse = torch.empty(w.q.shape[:3], dtype=torch.float32, device=dev) if with_lse else None

    def __call__(self, stream=None) -> int:
        w = self.w
        return B.pa_prefill_f16(self.p, w.q, w.k_buf, w.v_buf, self.out, self.lse, self.workspace, self.ws_bytes,
                                stream)

    def run(self, stream=None) -> torch.Tensor:
        B.check(self(stream), "prefill")
        return self.out

    def status(self, stream=None) -> int:
        st, flags = B.pa_read_status(self.workspace, stream)
        B.check(st, "pa_read_status")
        return flags
