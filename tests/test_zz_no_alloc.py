"""The allocation-free entry point (pa_decode_fp8_noalloc) against the
workspace entry point (pa_decode_fp8), through the C ABI on the GPU.

pa_decode_fp8_noalloc serves callers that cannot allocate device memory
themselves (code inside another framework's memory manager, latency-critical
host threads): its scratch is a fixed 16 MiB device array inside libpa.  Both
entry points run the same kernels with the same split plan, so their outputs
must agree bit for bit; one call is also checked against the FP64 oracle.
This file is collected last so that a failure here comes after every other
test has run; it also passes when run alone in a fresh process."""
import numpy as np
import pytest
import torch

from gpu_common import check_rows
from paged_gqa_decode_split_gb300 import binding as B
from paged_gqa_decode_split_gb300 import build as pa_build
from paged_gqa_decode_split_gb300 import decode as D
from paged_gqa_decode_split_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _noalloc(w, scales, out):
    """One pa_decode_fp8_noalloc call; allocates no torch memory itself."""
    p = D.params_for(w)
    kv = w.kv.data_ptr()
    st = B.pa_decode_fp8_noalloc(p, w.q, kv + w.k_offset, kv + w.v_offset, w.block_table, w.ctx_lens,
                                 scales.data_ptr(), scales.data_ptr() + 4, out)
    torch.cuda.synchronize()
    return st


def _scales(w):
    return torch.tensor([w.k_scale, w.v_scale], dtype=torch.float32, device=w.q.device)


def _same_bits(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pa_build.build()
    B.load()


def test_noalloc_matches_workspace_entry_on_two_calls():
    # two different workloads back to back on the shared scratch, then the first again
    first = wl.generate(wl.SPECS["b8_l128k"], wl.working_set_seed("b8_l128k", 5), device="cuda")
    second = wl.generate(wl.SPECS["b4_l32k"], wl.working_set_seed("b4_l32k", 2), device="cuda")
    for i, w in enumerate((first, second, first)):
        assert B.pa_decode_fp8_workspace_bytes(D.params_for(w)) <= B.PA_NOALLOC_SCRATCH_BYTES
        ref = D.Decoder(w).run().clone()
        out = torch.full_like(w.q, float("nan"))
        assert _noalloc(w, _scales(w), out) == B.PA_OK
        assert _same_bits(out, ref), f"call {i}: differs from pa_decode_fp8"
        if i == 1:
            # and against the oracle on sampled rows (each request's first and
            # last verify query of its first and last head, plus random rows)
            s = w.spec
            per = s.q_len * s.num_q_heads
            rng = np.random.default_rng(3)
            rows = set()
            for b in range(s.batch):
                rows |= {b * per, b * per + s.num_q_heads - 1, (b + 1) * per - s.num_q_heads, (b + 1) * per - 1}
                rows |= set((b * per + rng.integers(0, per, 4)).tolist())
            check_rows(w, out, np.array(sorted(rows), dtype=np.int32))
    # a geometry whose workspace exceeds the scratch is rejected before anything runs
    big = wl.generate(wl.SPECS["b16_mixed"], wl.working_set_seed("b16_mixed", 2), device="cuda")
    assert B.pa_decode_fp8_workspace_bytes(D.params_for(big)) > B.PA_NOALLOC_SCRATCH_BYTES
    out = torch.full_like(big.q, 7.0)
    assert _noalloc(big, _scales(big), out) == B.PA_ERR_WORKSPACE
    assert torch.all(out == 7.0)


def test_noalloc_allocates_nothing_after_warm_up():
    """After one warm-up call (which may load the scratch array's module), a
    further call leaves the device's free memory unchanged."""
    w = wl.generate(wl.SPECS["b4_l32k"], wl.working_set_seed("b4_l32k", 4), device="cuda")
    scales = _scales(w)
    out = torch.empty_like(w.q)
    assert _noalloc(w, scales, out) == B.PA_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert _noalloc(w, scales, out) == B.PA_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"


def test_noalloc_bad_input_does_not_carry_over():
    """A call with an invalid length zeroes that request's rows; the next
    valid call on the same shared scratch must equal the workspace entry
    point bit for bit (the per-request flags are cleared every call)."""
    w = wl.generate(wl.SPECS["b4_l32k"], wl.working_set_seed("b4_l32k", 6), device="cuda")
    scales = _scales(w)
    out = torch.full_like(w.q, float("nan"))
    good = w.ctx_lens.clone()
    w.ctx_lens[2] = w.spec.max_ctx_len + 1
    assert _noalloc(w, scales, out) == B.PA_OK
    assert torch.all(out[2] == 0) and not torch.signbit(out[2].float()).any()
    w.ctx_lens.copy_(good)
    out.fill_(float("nan"))
    assert _noalloc(w, scales, out) == B.PA_OK
    ref = D.Decoder(w).run().clone()
    assert _same_bits(out, ref)
