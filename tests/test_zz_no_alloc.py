"""The allocation-free entry point (pa_decode_fp8_noalloc) against the
workspace entry point (pa_decode_fp8), through the C ABI on the GPU.

pa_decode_fp8_noalloc serves callers that cannot allocate device memory
themselves (code inside another framework's memory manager, latency-critical
host threads): its scratch is a fixed 16 MiB device array inside libpa.  This
file is collected last so that a failure here comes after every other test
has run; it also passes when run alone in a fresh process."""
import numpy as np
import pytest
import torch

from paged_gqa_decode_split_gb300 import binding as B
from paged_gqa_decode_split_gb300 import build as pa_build
from paged_gqa_decode_split_gb300 import decode as D
from paged_gqa_decode_split_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-3
REL_L2 = 3e-3


def _noalloc(w, out):
    p = D.params_for(w)
    scales = torch.tensor([w.k_scale, w.v_scale], dtype=torch.float32, device=w.q.device)
    kv = w.kv.data_ptr()
    st = B.pa_decode_fp8_noalloc(p, w.q, kv + w.k_offset, kv + w.v_offset, w.block_table, w.ctx_lens,
                                 scales.data_ptr(), scales.data_ptr() + 4, out)
    torch.cuda.synchronize()
    return st


def _close(got, ref):
    g = got.float().cpu().numpy().astype(np.float64)
    r = ref.float().cpu().numpy().astype(np.float64)
    d = g - r
    assert np.all(np.isfinite(g))
    assert np.abs(d).max() <= MAX_ABS
    assert np.linalg.norm(d) <= REL_L2 * max(np.linalg.norm(r), 1e-30)


def test_noalloc_matches_workspace_entry_on_two_calls():
    pa_build.build()
    B.load()
    # two different workloads back to back on the shared scratch, then one twice
    first = wl.generate(wl.SPECS["b8_l128k"], wl.working_set_seed("b8_l128k", 5), device="cuda")
    second = wl.generate(wl.SPECS["b4_l32k"], wl.working_set_seed("b4_l32k", 2), device="cuda")
    for w in (first, second, first):
        assert B.pa_decode_fp8_workspace_bytes(D.params_for(w)) <= B.PA_NOALLOC_SCRATCH_BYTES
        ref = D.Decoder(w).run().clone()
        out = torch.full_like(w.q, float("nan"))
        assert _noalloc(w, out) == B.PA_OK
        _close(out, ref)
    # a geometry whose workspace exceeds the scratch is rejected before anything runs
    big = wl.generate(wl.SPECS["b16_mixed"], wl.working_set_seed("b16_mixed", 2), device="cuda")
    assert B.pa_decode_fp8_workspace_bytes(D.params_for(big)) > B.PA_NOALLOC_SCRATCH_BYTES
    out = torch.full_like(big.q, 7.0)
    assert _noalloc(big, out) == B.PA_ERR_WORKSPACE
    assert torch.all(out == 7.0)
