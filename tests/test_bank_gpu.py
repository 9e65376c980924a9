"""Workspace bank on the GPU: CUDA graphs captured for descending and for
growing batch sizes on bank panels, replayed after the bank grew and after
their inputs changed in place, match independent single-request calls bit for
bit ("DFlash2 concurrent long-context attention", section "Operator
validation": graphs captured for growing and descending batch sizes replay
after the bank was reused or grown, bitwise equal to independent requests)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_common import check_full
from paged_gqa_decode_split_gb300 import binding as B
from paged_gqa_decode_split_gb300 import build as pa_build
from paged_gqa_decode_split_gb300 import decode as D
from paged_gqa_decode_split_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pa_build.build()
    B.load()


def _prefix(w: wl.Workload, b: int) -> wl.Workload:
    """The first b requests of w as a batch of b (own Q, block table and
    lengths; the same KV pool)."""
    s = w.spec
    spec = wl.Spec(f"{s.name}_b{b}", s.kind, b, s.num_kv_heads, s.num_q_heads, s.head_dim, s.q_len, s.page_size,
                   s.max_ctx_len, ctx_lens=(0,) * b, layout=s.layout, base_pad=s.base_pad)
    return wl.Workload(spec=spec, q=w.q[:b].clone(), kv=w.kv, k_offset=w.k_offset, v_offset=w.v_offset,
                       k_strides=w.k_strides, v_strides=w.v_strides, block_table=w.block_table[:b].clone(),
                       ctx_lens=w.ctx_lens[:b].clone(), num_pages=w.num_pages, k_scale=w.k_scale,
                       v_scale=w.v_scale)


def _capture(dec: D.Decoder, stream: torch.cuda.Stream) -> torch.cuda.CUDAGraph:
    # the panel, the scales and the inputs were written on the current stream
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        B.check(dec(stream), "eager call")
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        B.check(dec(stream), "captured call")
    return g


def _singles(w: wl.Workload) -> torch.Tensor:
    """Each request alone, with its own workspace."""
    outs = []
    for b in range(w.spec.batch):
        outs.append(D.Decoder(_prefix_one(w, b)).run().clone())
    torch.cuda.synchronize()
    return torch.cat(outs)


def _prefix_one(w: wl.Workload, b: int) -> wl.Workload:
    s = w.spec
    spec = wl.Spec(f"{s.name}_r{b}", s.kind, 1, s.num_kv_heads, s.num_q_heads, s.head_dim, s.q_len, s.page_size,
                   s.max_ctx_len, ctx_lens=(0,), layout=s.layout, base_pad=s.base_pad)
    return wl.Workload(spec=spec, q=w.q[b:b + 1].clone(), kv=w.kv, k_offset=w.k_offset, v_offset=w.v_offset,
                       k_strides=w.k_strides, v_strides=w.v_strides, block_table=w.block_table[b:b + 1].clone(),
                       ctx_lens=w.ctx_lens[b:b + 1].clone(), num_pages=w.num_pages, k_scale=w.k_scale,
                       v_scale=w.v_scale)


def test_graphs_across_batch_sizes_share_and_grow_the_bank():
    spec = wl.Spec("bank", "fp8", 16, 1, 6, 256, 8, 64, 6000, ctx_range=(0, 6000), zero_slots=(5,))
    w = wl.generate(spec, 77, device="cuda")
    bank = D.WorkspaceBank()
    s_desc, s_grow = torch.cuda.Stream(), torch.cuda.Stream()
    runs = []  # (workload, decoder, graph, stream)
    # descending batch sizes on one stream: one panel
    for b in (16, 8, 4):
        wb = _prefix(w, b)
        dec = D.Decoder(wb, bank=bank, stream=s_desc)
        runs.append((wb, dec, _capture(dec, s_desc), s_desc))
    assert bank.stats()[0] == 1
    assert len({r[1].workspace for r in runs}) == 1
    # growing batch sizes on another stream: a new panel for every growth
    for b in (2, 8, 16):
        wb = _prefix(w, b)
        dec = D.Decoder(wb, bank=bank, stream=s_grow)
        runs.append((wb, dec, _capture(dec, s_grow), s_grow))
    assert bank.stats()[0] == 4
    assert len({r[1].workspace for r in runs[3:]}) == 3
    assert not {r[1].workspace for r in runs[3:]} & {runs[0][1].workspace}
    # a later small batch on the grown stream gets the largest panel
    assert D.Decoder(_prefix(w, 2), bank=bank, stream=s_grow).workspace == runs[-1][1].workspace

    # change every captured input in place (Q; lengths, with a zero row, kept
    # within the pages each request's block-table row holds), replay the older
    # graphs after the bank grew, and compare bit for bit
    gen = torch.Generator(device="cuda").manual_seed(5)
    for k, (wb, dec, g, st) in enumerate(runs):
        wb.q.copy_(torch.randn(wb.q.shape, generator=gen, device="cuda").half())
        old = wb.ctx_lens.clone()
        frac = torch.rand(wb.spec.batch, generator=gen, device="cuda")
        new = torch.minimum((frac * (old.float() + 1)).floor().to(torch.int32), old)
        if k % 2:
            new[0] = 0
        wb.ctx_lens.copy_(new)
    torch.cuda.synchronize()
    for wb, dec, g, st in runs:
        with torch.cuda.stream(st):
            g.replay()
    torch.cuda.synchronize()
    for wb, dec, g, st in runs:
        assert dec.status() == 0
        ref = _singles(wb)
        assert torch.equal(dec.out.view(torch.int16), ref.view(torch.int16)), wb.spec.name
    check_full(runs[0][0], runs[0][1].out)
    bank.close()
