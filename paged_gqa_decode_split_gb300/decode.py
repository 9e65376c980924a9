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


class WorkspaceBank:
    """pa_bank over torch device memory: every panel is a zero-filled uint8
    tensor held here until close() (or until the bank is garbage collected).
    Grow the bank outside CUDA-graph capture (an eager call first), so that no
    panel comes from a capture's private memory pool."""

    def __init__(self):
        self._held: dict[int, torch.Tensor] = {}

        def alloc(nbytes: int, device: int) -> int:
            t = torch.zeros(nbytes + 256, dtype=torch.uint8, device=torch.device("cuda", device))
            ptr = (t.data_ptr() + 255) & ~255
            self._held[ptr] = t
            return ptr

        def free(ptr: int, nbytes: int, device: int) -> None:
            self._held.pop(ptr, None)

        self.handle, self._keepalive = B.pa_bank_create(alloc, free)
        if not self.handle:
            raise RuntimeError("pa_bank_create failed")

    def workspace(self, p: B.pa_params, device: int, stream=None) -> tuple[int, int]:
        st, ptr, nbytes = B.pa_bank_workspace(self.handle, p, device, stream)
        B.check(st, "pa_bank_workspace")
        return ptr, nbytes

    def stats(self) -> tuple[int, int]:
        st, panels, nbytes = B.pa_bank_stats(self.handle)
        B.check(st, "pa_bank_stats")
        return panels, nbytes

    def close(self) -> None:
        if self.handle:
            B.check(B.pa_bank_destroy(self.handle), "pa_bank_destroy")
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Decoder:
    """Holds the device-side buffers one workload needs (output, workspace,
    scales) and enqueues the decode call of its kind on a stream:
    pa_decode_fp8 ("fp8"), pa_decode_e5m2 ("e5m2"), pa_decode_f16 ("f16"),
    pa_decode_bf16_d128 / pa_decode_bf16_d256 ("bf16", head_dim 128 / 256)."""

    def __init__(self, w: Workload, *, with_lse: bool = False, bank: "WorkspaceBank | None" = None, stream=None):
        if not w.q.is_cuda:
            raise ValueError("the workload must be on a CUDA device")
        self.w = w
        self.p = params_for(w)
        s = w.spec
        dev = w.q.device
        self.kind = s.kind
        self.fp8 = s.kind in ("fp8", "e5m2")   # 8-bit K/V with per-tensor scales
        nbytes = (B.pa_decode_bf16_d128_workspace_bytes(self.p) if s.head_dim == 128 else
                  B.pa_decode_fp8_workspace_bytes(self.p))
        if nbytes == 0:
            raise ValueError("libpa rejects this geometry")
        if bank is not None:
            # a panel shared with every other decoder of this (device, stream,
            # contract); such decoders must be called on `stream` only
            index = dev.index if dev.index is not None else torch.cuda.current_device()
            self.workspace, self.ws_bytes = bank.workspace(self.p, index, stream)
        else:
            self.ws_bytes = nbytes
            self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        self.out = torch.empty_like(w.q)
        self.lse = (torch.empty(w.q.shape[:3], dtype=torch.float32, device=dev) if (with_lse and s.kind == "bf16")
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
        if self.kind == "f16":
            return B.pa_decode_f16(self.p, w.q, kv + w.k_offset, kv + w.v_offset, w.block_table, w.ctx_lens,
                                   self.out, self.workspace, self.ws_bytes, stream)
        fn = B.pa_decode_bf16_d128 if w.spec.head_dim == 128 else B.pa_decode_bf16_d256
        return fn(self.p, w.q, kv + w.k_offset, kv + w.v_offset, w.block_table, w.ctx_lens, self.out, self.lse,
                  self.workspace, self.ws_bytes, stream)

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
