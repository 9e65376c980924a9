"""Convenience calls over the C ABI for workloads held in torch tensors.

Device memory (output, workspace, scale scalars) is allocated with torch; the
arithmetic runs in libpa's kernels through ``binding``."""
from __future__ import annotations

import torch

from . import binding as B
from .workloads import Workload


def params_for(w: Workload) -> B.pa_params:
    s = w.spec
    return B.make_params(batch=s.batch, num_kv_heads=s.num_kv_heads, num_q_heads=s.num_q_heads,
                         head_dim=s.head_dim, q_len=s.q_len, page_size=s.page_size,
                         max_pages_per_req=w.block_table.shape[1], num_pages=w.num_pages,
                         max_ctx_len=s.max_ctx_len, k_strides=w.k_strides, v_strides=w.v_strides)


class Decoder:
    """Holds the device-side buffers one workload needs (output, workspace,
    scales) and enqueues pa_decode_fp8 / pa_decode_e5m2 / pa_decode_bf16_d128 on
    a stream."""

    def __init__(self, w: Workload, *, with_lse: bool = False):
        if not w.q.is_cuda:
            raise ValueError("the workload must be on a CUDA device")
        self.w = w
        self.p = params_for(w)
        s = w.spec
        dev = w.q.device
        self.kind = s.kind
        self.fp8 = s.kind in ("fp8", "e5m2")   # 8-bit K/V with per-tensor scales
        nbytes = (B.pa_decode_fp8_workspace_bytes(self.p) if self.fp8 else
                  B.pa_decode_bf16_d128_workspace_bytes(self.p))
        if nbytes == 0:
            raise ValueError("libpa rejects this geometry")
        self.ws_bytes = nbytes
        self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        self.out = torch.empty_like(w.q)
        self.lse = (torch.empty(w.q.shape[:3], dtype=torch.float32, device=dev) if (with_lse and not self.fp8)
                    else None)
        self.scales = torch.tensor([w.k_scale, w.v_scale], dtype=torch.float32, device=dev)

    def set_workload(self, w: Workload) -> None:
        """Point the decoder at another workload of the same geometry (new
        tensors, lengths and scales; same shapes)."""
        self.w = w
        self.p = params_for(w)
        self.scales.copy_(torch.tensor([w.k_scale, w.v_scale], dtype=torch.float32))

    def __call__(self, stream=None) -> int:
        w = self.w
        kv = w.kv.data_ptr()
        if self.fp8:
            fn = B.pa_decode_fp8 if self.kind == "fp8" else B.pa_decode_e5m2
            return fn(self.p, w.q, kv + w.k_offset, kv + w.v_offset, w.block_table, w.ctx_lens,
                      self.scales.data_ptr(), self.scales.data_ptr() + 4, self.out, self.workspace, self.ws_bytes,
                      stream)
        return B.pa_decode_bf16_d128(self.p, w.q, kv + w.k_offset, kv + w.v_offset, w.block_table, w.ctx_lens,
                                     self.out, self.lse, self.workspace, self.ws_bytes, stream)

    def run(self, stream=None) -> torch.Tensor:
        B.check(self(stream), "decode")
        return self.out

    def status(self, stream=None) -> int:
        st, flags = B.pa_read_status(self.workspace, stream)
        B.check(st, "pa_read_status")
        return flags


def decode(w: Workload, *, with_lse: bool = False):
    """One decode call on the current stream; returns out (and lse for bf16)."""
    d = Decoder(w, with_lse=with_lse)
    d.run()
    return (d.out, d.lse) if with_lse else d.out
