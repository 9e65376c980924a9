"""Test helpers: hand one seeded workload to the FP64 oracle, and build dense
references with independent library routines (torch casts, float64 SDPA)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_gqa_decode_split_gb300 import workloads as wl


def q_bits(w: wl.Workload) -> np.ndarray:
    return w.q.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def run_oracle(w: wl.Workload, rows=None, lib=None, num_threads: int = 0):
    """Evaluate the FP64 oracle on workload w (all rows, or the listed flat rows)."""
    s = w.spec
    return oracle.paged_attn(
        s.kind, q=q_bits(w), kv=w.kv.detach().cpu().numpy(), k_offset=w.k_offset, v_offset=w.v_offset,
        k_strides=w.k_strides, v_strides=w.v_strides, block_table=w.block_table.cpu().numpy(),
        ctx_lens=w.ctx_lens.cpu().numpy(), num_kv_heads=s.num_kv_heads, page_size=s.page_size,
        k_scale=w.k_scale, v_scale=w.v_scale, rows=rows, num_threads=num_threads, lib=lib)


def _elements(w: wl.Workload, which: str, b: int, g: int, n: int) -> torch.Tensor:
    """Dense float64 K or V rows 0..n-1 of request b, KV head g, decoded with
    torch's own float8_e4m3fn / float8_e5m2 / float16 / bfloat16 casts (not the
    oracle's decoders)."""
    s = w.spec
    kv = w.kv.detach().cpu()
    off = w.k_offset if which == "k" else w.v_offset
    st = w.k_strides if which == "k" else w.v_strides
    row_bytes = s.head_dim * s.elem_bytes
    bt = w.block_table.cpu()
    rows = []
    for j in range(n):
        page = int(bt[b, j // s.page_size])
        start = off + page * st[0] + (j % s.page_size) * st[1] + g * st[2]
        rows.append(kv[start:start + row_bytes])
    if not rows:
        return torch.zeros((0, s.head_dim), dtype=torch.float64)
    raw = torch.stack(rows)
    if s.kind in ("fp8", "e5m2"):
        scale = w.k_scale if which == "k" else w.v_scale
        dtype = torch.float8_e4m3fn if s.kind == "fp8" else torch.float8_e5m2
        return raw.view(dtype).to(torch.float64) * torch.tensor(scale, dtype=torch.float32).double()
    return raw.view(torch.bfloat16 if s.kind == "bf16" else torch.float16).to(torch.float64)


def dense_reference(w: wl.Workload):
    """float64 reference through torch.nn.functional.scaled_dot_product_attention
    with an explicit boolean causal mask; rows with no key come back as None."""
    s = w.spec
    B, q_len, Hq, D = s.batch, s.q_len, s.num_q_heads, s.head_dim
    G = Hq // s.num_kv_heads
    q = w.q.detach().cpu().to(torch.float64)
    out = np.full((B, q_len, Hq, D), np.nan)
    lse = np.full((B, q_len, Hq), np.nan)
    for b in range(B):
        L = int(w.ctx_lens[b])
        for g in range(s.num_kv_heads):
            if L <= 0:
                continue
            K = _elements(w, "k", b, g, L)
            V = _elements(w, "v", b, g, L)
            j = torch.arange(L)
            qi = torch.arange(q_len)
            mask = j[None, :] <= (L - q_len + qi)[:, None]          # [q_len, L]
            for hl in range(G):
                h = g * G + hl
                qs = q[b, :, h, :]                                   # [q_len, D]
                o = torch.nn.functional.scaled_dot_product_attention(
                    qs[None, None], K[None, None], V[None, None], attn_mask=mask[None, None])[0, 0]
                scores = (qs @ K.T) / np.sqrt(D)
                scores = scores.masked_fill(~mask, float("-inf"))
                ls = torch.logsumexp(scores, dim=-1)
                for i in range(q_len):
                    if bool(mask[i].any()):
                        out[b, i, h] = o[i].numpy()
                        lse[b, i, h] = float(ls[i])
    return out, lse


def visible(w: wl.Workload) -> np.ndarray:
    """Boolean [B, q_len, Hq]: rows that see at least one key."""
    s = w.spec
    L = w.ctx_lens.cpu().numpy()[:, None, None]
    qi = np.arange(s.q_len)[None, :, None]
    return np.broadcast_to(L - s.q_len + qi + 1 > 0, (s.batch, s.q_len, s.num_q_heads))
