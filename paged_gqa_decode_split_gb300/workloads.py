"""Seeded synthetic inputs for paged GQA decode / speculative-verify attention.

This module draws random inputs and lays them out in paged form.  It holds none
of the attention arithmetic: the CUDA path and the FP64 oracle both consume
what it produces, and neither is imported here.

Workload shapes follow the pages' validation and timing fixtures:
  * "DFlash2 concurrent long-context attention", sections "Operator
    validation" (B2/B4/B8/B16, contexts 3297 .. 262144, pages 1024/1536/1648/
    3296, interleaved and eight-byte-only aligned KV strides, padded requests
    and zero-length rows) and "Attention-only measurements" (q8 verify,
    page 1648, contexts 32768 and 131072 at 4 and 8 concurrent requests,
    16 independent per-layer KV working sets).
  * "perf(fa2): port decode GQA group-swap into d128 varlen launcher" (vllm.cpp
    pull request #48), description: BF16 head-dim-128 decode with GQA ratio
    4 (32 query heads over 8 KV heads), batch 1/2/4/8, paged KV.

Value recipe: Q ~ N(0, 1) in FP16 (BF16 for d128).  K and V ~ N(0, 1) drawn in
FP32; for E4M3 each of K and V gets one FP32 scale amax/448 and the bytes are
clamp(x / scale, -448, 448) cast to E4M3 with round-to-nearest-even by torch's
float8_e4m3fn conversion.  E5M2 K/V (a cache type that keeps its own graph
set beside E4M3: "DFlash2 concurrent long-context attention", section "Why the
single-request optimization was missing from concurrent decode") follows the
same recipe with the format's largest finite value, 57344, in place of 448 and
torch's float8_e5m2 conversion.  FP16 and BF16 K/V (16-bit caches, no
scales) are the N(0, 1) draws rounded to the element type.  Pages are assigned to requests through a random
permutation of the pool; block-table entries past a request's last page are -1
and must never be read.  Padded batch slots have ctx_len 0, Q = NaN and a block
table row of -1.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

E4M3_MAX = 448.0
E5M2_MAX = 57344.0


@dataclasses.dataclass(frozen=True)
class Spec:
    """Shape and structure of one workload (values are drawn by ``generate``)."""

    name: str
    kind: str                      # "fp8": FP16 Q + E4M3 K/V, "e5m2": FP16 Q + E5M2 K/V,
                                   # "f16": FP16 Q/K/V, "bf16": BF16 Q/K/V
    batch: int
    num_kv_heads: int
    num_q_heads: int
    head_dim: int
    q_len: int
    page_size: int
    max_ctx_len: int               # host bound: block-table width and workspace
    ctx_lens: Optional[Sequence[int]] = None   # explicit lengths, or drawn below
    ctx_range: Optional[tuple[int, int]] = None  # uniform integer lengths in [lo, hi]
    zero_slots: Sequence[int] = ()             # live slots forced to length 0
    padded_slots: Sequence[int] = ()           # padded slots: length 0, Q = NaN
    layout: str = "separate"       # "separate": K pages then V pages; "interleaved": [.., Hkv, 2, D];
                                   # "padded_tokens": separate, each slot's Hkv rows followed by 8 unused
                                   # bytes (token strides 8 past a multiple of 16)
    base_pad: int = 0              # byte offset of the K/V base (8 gives 8-byte-only alignment)
    extra_pages: int = 0           # unused pages in the pool

    @property
    def elem_bytes(self) -> int:
        return 1 if self.kind in ("fp8", "e5m2") else 2

    @property
    def max_pages_per_req(self) -> int:
        return max(1, math.ceil(self.max_ctx_len / self.page_size))


@dataclasses.dataclass
class Workload:
    spec: Spec
    q: torch.Tensor             # [B, q_len, Hq, D] float16 (fp8 kind) or bfloat16
    kv: torch.Tensor            # flat uint8 buffer with K and V pages
    k_offset: int               # byte offset of K (page 0, slot 0, head 0, d 0) in kv
    v_offset: int
    k_strides: tuple[int, int, int]   # (page, slot, head) strides in bytes
    v_strides: tuple[int, int, int]
    block_table: torch.Tensor   # int32 [B, max_pages_per_req]
    ctx_lens: torch.Tensor      # int32 [B]
    num_pages: int
    k_scale: float = 1.0        # FP32 values (E4M3 only)
    v_scale: float = 1.0

    def to(self, device) -> "Workload":
        return dataclasses.replace(self, q=self.q.to(device), kv=self.kv.to(device),
                                   block_table=self.block_table.to(device), ctx_lens=self.ctx_lens.to(device))

    def unique_kv_bytes(self) -> int:
        """Bytes of K and V that the definition touches: every visible key of
        every request, once per KV head (page tails, Q, output excluded)."""
        s = self.spec
        return int(sum(int(L) for L in self.ctx_lens.tolist())) * s.num_kv_heads * s.head_dim * s.elem_bytes * 2


# The five configurations the pages' fixtures describe.
SPECS: dict[str, Spec] = {
    "b1_l3297": Spec("b1_l3297", "fp8", 1, 1, 6, 256, 8, 1648, 3297, ctx_lens=(3297,)),
    "b4_l32k": Spec("b4_l32k", "fp8", 4, 1, 6, 256, 8, 1648, 32768, ctx_lens=(32768,) * 4),
    "b8_l128k": Spec("b8_l128k", "fp8", 8, 1, 6, 256, 8, 1648, 131072, ctx_lens=(131072,) * 8),
    "b16_mixed": Spec("b16_mixed", "fp8", 16, 2, 12, 256, 8, 3296, 262144, ctx_range=(0, 262144),
                      zero_slots=(4, 9), padded_slots=(13, 14, 15), layout="interleaved", base_pad=8),
}
# E5M2, FP16 and BF16 K/V on the E4M3 configurations' shapes
for _n in ("b1_l3297", "b8_l128k"):
    for _k in ("e5m2", "f16", "bf16"):
        SPECS[f"{_n}_{_k}"] = dataclasses.replace(SPECS[_n], name=f"{_n}_{_k}", kind=_k)
for _b in (1, 2, 4, 8):
    SPECS[f"d128_b{_b}"] = Spec(f"d128_b{_b}", "bf16", _b, 8, 32, 128, 1, 16, 32768, ctx_range=(1024, 32768))

CONFIG_SEED = {"b1_l3297": 1000, "b4_l32k": 1001, "b8_l128k": 1002, "b16_mixed": 1003,
               "d128_b1": 1004, "d128_b2": 1014, "d128_b4": 1024, "d128_b8": 1034,
               "b1_l3297_e5m2": 1005, "b8_l128k_e5m2": 1006, "b1_l3297_f16": 1007, "b8_l128k_f16": 1008,
               "b1_l3297_bf16": 1009, "b8_l128k_bf16": 1010}


def working_set_seed(name: str, w: int) -> int:
    """Seed of per-layer working set ``w`` of configuration ``name``."""
    return CONFIG_SEED.get(name, 1000) + 97 * w


def _draw_lengths(spec: Spec, gen: torch.Generator) -> list[int]:
    if spec.ctx_lens is not None:
        lens = [int(x) for x in spec.ctx_lens]
    else:
        lo, hi = spec.ctx_range
        lens = torch.randint(lo, hi + 1, (spec.batch,), generator=gen).tolist()
    for i in list(spec.zero_slots) + list(spec.padded_slots):
        lens[i] = 0
    if len(lens) != spec.batch:
        raise ValueError("ctx_lens length must equal batch")
    if max(lens) > spec.max_ctx_len:
        raise ValueError("a context length exceeds max_ctx_len")
    return lens


def _quantize(x: torch.Tensor, kind: str) -> tuple[torch.Tensor, float]:
    """FP32 tensor -> (8-bit codes as uint8, FP32 per-tensor scale amax/fmax),
    fmax = 448 for E4M3 ("fp8"), 57344 for E5M2."""
    fmax, dtype = (E4M3_MAX, torch.float8_e4m3fn) if kind == "fp8" else (E5M2_MAX, torch.float8_e5m2)
    amax = x.abs().max().to(torch.float32)
    scale = (amax / fmax).clamp_min(torch.finfo(torch.float32).tiny)
    codes = (x / scale).clamp(-fmax, fmax).to(dtype)
    return codes.view(torch.uint8), float(scale.item())


def generate(spec: Spec, seed: int, device: str | torch.device = "cpu",
             ctx_lens: Optional[Sequence[int]] = None) -> Workload:
    """Draw one seeded workload of shape ``spec`` on ``device``.

    ``ctx_lens`` overrides the spec's lengths (used for edge-case tests).
    Random draws happen on ``device``; a CPU and a CUDA draw with the same seed
    differ, so a test hands the same tensors to both sides.
    """
    device = torch.device(device)
    cpu_gen = torch.Generator(device="cpu").manual_seed(seed)
    gen = torch.Generator(device=device).manual_seed(seed + 1)
    lens = list(ctx_lens) if ctx_lens is not None else _draw_lengths(spec, cpu_gen)
    B, Hkv, Hq, D, ps = spec.batch, spec.num_kv_heads, spec.num_q_heads, spec.head_dim, spec.page_size
    if Hq % Hkv:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    pages_per_req = [math.ceil(L / ps) for L in lens]
    num_pages = max(1, sum(pages_per_req) + spec.extra_pages)
    mpr = spec.max_pages_per_req
    # random page assignment
    perm = torch.randperm(num_pages, generator=cpu_gen)
    bt = torch.full((B, mpr), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages_per_req):
        bt[b, :n] = perm[off:off + n].to(torch.int32)
        off += n
    # queries
    qdtype = torch.bfloat16 if spec.kind == "bf16" else torch.float16
    q = torch.randn((B, spec.q_len, Hq, D), generator=gen, device=device, dtype=torch.float32).to(qdtype)
    for i in spec.padded_slots:
        q[i] = float("nan")
    # K and V pages, logical shape [num_pages, ps, Hkv, D]
    shape = (num_pages, ps, Hkv, D)
    kx = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if spec.kind in ("fp8", "e5m2"):
        kb, k_scale = _quantize(kx, spec.kind)
        del kx
        vx = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        vb, v_scale = _quantize(vx, spec.kind)
        del vx
    else:
        edt = torch.bfloat16 if spec.kind == "bf16" else torch.float16
        kb = kx.to(edt).view(torch.uint8).reshape(*shape[:3], D * 2)
        del kx
        vb = torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(edt)
        vb = vb.view(torch.uint8).reshape(*shape[:3], D * 2)
        k_scale = v_scale = 1.0
    row = D * spec.elem_bytes
    pad = spec.base_pad
    if spec.layout == "separate":
        region = num_pages * ps * Hkv * row
        kv = torch.zeros(pad + 2 * region + 16, dtype=torch.uint8, device=device)
        kv[pad:pad + region] = kb.reshape(-1)
        kv[pad + region:pad + 2 * region] = vb.reshape(-1)
        strides = (ps * Hkv * row, Hkv * row, row)
        k_off, v_off = pad, pad + region
        k_str = v_str = strides
    elif spec.layout == "interleaved":
        total = num_pages * ps * Hkv * 2 * row
        kv = torch.zeros(pad + total + 16, dtype=torch.uint8, device=device)
        view = kv[pad:pad + total].view(num_pages, ps, Hkv, 2, row)
        view[:, :, :, 0, :] = kb.reshape(num_pages, ps, Hkv, row)
        view[:, :, :, 1, :] = vb.reshape(num_pages, ps, Hkv, row)
        strides = (ps * Hkv * 2 * row, Hkv * 2 * row, 2 * row)
        k_off, v_off = pad, pad + row
        k_str = v_str = strides
    elif spec.layout == "padded_tokens":
        tstride = Hkv * row + 8
        region = num_pages * ps * tstride
        kv = torch.zeros(pad + 2 * region + 16, dtype=torch.uint8, device=device)
        for off, src in ((pad, kb), (pad + region, vb)):
            view = kv[off:off + region].view(num_pages, ps, tstride)
            view[:, :, :Hkv * row] = src.reshape(num_pages, ps, Hkv * row)
        strides = (ps * tstride, tstride, row)
        k_off, v_off = pad, pad + region
        k_str = v_str = strides
    else:
        raise ValueError(spec.layout)
    return Workload(spec=spec, q=q, kv=kv, k_offset=k_off, v_offset=v_off, k_strides=k_str, v_strides=v_str,
                    block_table=bt.to(device), ctx_lens=torch.tensor(lens, dtype=torch.int32, device=device),
                    num_pages=num_pages, k_scale=k_scale, v_scale=v_scale)


def small_spec(kind: str = "fp8", *, batch: int = 2, num_kv_heads: int = 1, group: int = 6, q_len: int = 8,
               page_size: int = 16, max_ctx_len: int = 64, layout: str = "separate", base_pad: int = 0,
               head_dim: Optional[int] = None, name: str = "small") -> Spec:
    """A small spec for tests (lengths are passed to ``generate``)."""
    D = head_dim or (128 if kind == "bf16" else 256)
    return Spec(name, kind, batch, num_kv_heads, num_kv_heads * group, D, q_len, page_size, max_ctx_len,
                ctx_lens=(0,) * batch, layout=layout, base_pad=base_pad)


# ------------------------------------------------------------------ prefill --
# Causal long prefill ("SM70 attention and quantized projection coverage
# across TP sizes", sections "Accumulation audit and rejected tuning" and
# "Graph replay and long-prefill follow-up": Q8192 x KV262144, GQA 6 with
# Hkv 1/2/4, B1/B2, FP16 inputs, random values).  Q, K and V ~ N(0, 1) drawn
# in FP32 and rounded to FP16.  K and V are dense per request
# ([B][kv_len][Hkv][256], or with `token_pad` unused elements after each
# token's Hkv rows to exercise the strides).

@dataclasses.dataclass(frozen=True)
class PrefillSpec:
    name: str
    batch: int
    q_len: int
    kv_len: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int = 256
    token_pad: int = 0  # extra FP16 elements after each token's Hkv rows (a multiple of 8)


@dataclasses.dataclass
class PrefillWorkload:
    spec: PrefillSpec
    q: torch.Tensor        # FP16 [B][q_len][Hq][D]
    k_buf: torch.Tensor    # FP16 storage of K
    v_buf: torch.Tensor
    k_strides: tuple[int, int, int]  # (batch, token, head) in elements
    v_strides: tuple[int, int, int]

    def to(self, device) -> "PrefillWorkload":
        return dataclasses.replace(self, q=self.q.to(device), k_buf=self.k_buf.to(device),
                                   v_buf=self.v_buf.to(device))

    def key_view(self, which: str) -> torch.Tensor:
        """[B][kv_len][Hkv][D] strided view of K or V."""
        s = self.spec
        buf, st = (self.k_buf, self.k_strides) if which == "k" else (self.v_buf, self.v_strides)
        return buf.as_strided((s.batch, s.kv_len, s.num_kv_heads, s.head_dim), (*st, 1))


PREFILL_SPECS = {
    # the pages' single-GPU prefill operator at the TP4 local geometry (Hkv 1)
    "prefill_q8192_kv262144": PrefillSpec("prefill_q8192_kv262144", 1, 8192, 262144, 6, 1),
    # the TP2 / TP1 local geometries, B2 (the bitwise per-head check's shapes)
    "prefill_q8192_kv262144_hkv2_b2": PrefillSpec("prefill_q8192_kv262144_hkv2_b2", 2, 8192, 262144, 12, 2),
}
# the TP1 local geometry (Hkv 4, Hq 24) of the same page
PREFILL_SPECS["prefill_q8192_kv262144_hkv4"] = PrefillSpec("prefill_q8192_kv262144_hkv4", 1, 8192, 262144, 24, 4)
# a smaller case of the same kernel for profiler captures (K and V still exceed L2)
PREFILL_SPECS["prefill_q2048_kv131072"] = PrefillSpec("prefill_q2048_kv131072", 1, 2048, 131072, 6, 1)
PREFILL_SEED = {"prefill_q8192_kv262144": 2001, "prefill_q8192_kv262144_hkv2_b2": 2002, "prefill_q2048_kv131072": 2003,
                "prefill_q8192_kv262144_hkv4": 2004}


def generate_prefill(spec: PrefillSpec, seed: int, device: str | torch.device = "cpu") -> PrefillWorkload:
    """Draw one seeded prefill workload of shape ``spec`` on ``device``."""
    device = torch.device(device)
    gen = torch.Generator(device=device).manual_seed(seed)
    B, Q, KV, Hq, Hkv, D = spec.batch, spec.q_len, spec.kv_len, spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    if Hq % Hkv:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    if spec.token_pad % 8:
        raise ValueError("token_pad must be a multiple of 8 elements")
    q = torch.randn((B, Q, Hq, D), generator=gen, device=device, dtype=torch.float32).to(torch.float16)
    tstride = Hkv * D + spec.token_pad
    strides = (KV * tstride, tstride, D)
    bufs = []
    for _ in range(2):
        x = torch.randn((B, KV, Hkv, D), generator=gen, device=device, dtype=torch.float32).to(torch.float16)
        buf = torch.zeros(B * KV * tstride, dtype=torch.float16, device=device)
        buf.as_strided((B, KV, Hkv, D), (*strides, 1)).copy_(x)
        del x
        bufs.append(buf)
    return PrefillWorkload(spec=spec, q=q, k_buf=bufs[0], v_buf=bufs[1], k_strides=strides, v_strides=strides)
