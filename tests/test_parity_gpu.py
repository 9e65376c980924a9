"""GPU parity: the CUDA path through the C ABI against the FP64 oracle.

Small cases are compared row by row in full (several 128-key tiles, ragged
tails, every q_len, GQA up to 8, several KV heads, 8-byte-only aligned
interleaved K/V, zero-length and padded slots, contexts shorter than the verify
window); the workload configurations are run at full size in the same
launch configuration the benchmark uses and compared on all rows where the
oracle is affordable, otherwise on sampled rows."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_common import check_full, check_rows, to_f64
from paged_gqa_decode_split_gb300 import binding as B
from paged_gqa_decode_split_gb300 import build as pa_build
from paged_gqa_decode_split_gb300 import decode as D
from paged_gqa_decode_split_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pa_build.build()
    B.load()


def _small(kind, lens, *, Hkv=1, group=6, q_len=8, page_size=16, layout="separate", base_pad=0, seed=1,
           max_ctx=None, padded=(), D=None):
    D_ = D or (128 if kind == "bf16" else 256)
    spec = wl.Spec(f"small_{kind}", kind, len(lens), Hkv, Hkv * group, D_, q_len, page_size,
                   max_ctx or max(max(lens), 1), ctx_lens=tuple(lens), padded_slots=tuple(padded), layout=layout,
                   base_pad=base_pad)
    return wl.generate(spec, seed).to("cuda")


SMALL = [
    # id, kind, lens, kwargs
    ("fp8_tiles_tail", "fp8", [300, 37], {}),
    ("fp8_hkv2_interleaved_8B", "fp8", [700, 129, 0], dict(Hkv=2, page_size=32, layout="interleaved", base_pad=8)),
    ("fp8_q1", "fp8", [1000, 5], dict(q_len=1)),
    ("fp8_q2", "fp8", [513, 2], dict(q_len=2)),
    ("fp8_q3", "fp8", [257, 40], dict(q_len=3)),
    ("fp8_q5_hkv3", "fp8", [384, 128], dict(q_len=5, Hkv=3)),
    ("fp8_g8_q8", "fp8", [513, 64], dict(group=8)),
    ("fp8_g4_q4", "fp8", [640, 11], dict(group=4, q_len=4)),
    ("fp8_short_contexts", "fp8", [1, 2, 7, 8, 9, 16, 0], {}),
    ("fp8_page48_many_splits", "fp8", [20000, 4097], dict(page_size=48)),
    # TMA boxes of 64 + 16 slots per page piece, whole 128-slot boxes, and an
    # interleaved K/V layout that is 16-byte aligned (so loaded by TMA)
    ("fp8_page80_tma", "fp8", [1000, 333], dict(page_size=80)),
    ("fp8_page128_tma", "fp8", [2000, 129], dict(page_size=128)),
    ("fp8_interleaved_16B_tma", "fp8", [900, 257], dict(Hkv=2, page_size=64, layout="interleaved")),
    ("fp8_padded_nan", "fp8", [900, 0, 33, 0], dict(padded=(3,))),
    # E5M2 K/V: the TMA and the cp.async (8-byte aligned) loaders, several tile widths
    ("e5m2_tiles_tail", "e5m2", [300, 37], {}),
    ("e5m2_hkv2_interleaved_8B", "e5m2", [700, 129, 0], dict(Hkv=2, page_size=32, layout="interleaved", base_pad=8)),
    ("e5m2_q1", "e5m2", [1000, 5], dict(q_len=1)),
    ("e5m2_g8_page80_tma", "e5m2", [1000, 333], dict(group=8, page_size=80)),
    # 16-bit K/V at D 256 (512-byte rows, two staging fills per tile): TMA and
    # cp.async loaders, several tile widths
    ("f16_tiles_tail", "f16", [300, 37], {}),
    ("f16_hkv2_interleaved_8B", "f16", [700, 129, 0], dict(Hkv=2, page_size=32, layout="interleaved", base_pad=8)),
    ("f16_q1_page80_tma", "f16", [1000, 5], dict(q_len=1, page_size=80)),
    ("f16_g8", "f16", [513, 64], dict(group=8)),
    ("bf16_d256_tiles_tail", "bf16", [300, 37], dict(D=256)),
    ("bf16_d256_hkv2_interleaved_8B", "bf16", [700, 129, 0],
     dict(D=256, Hkv=2, page_size=32, layout="interleaved", base_pad=8)),
    ("bf16_d256_g4_q1", "bf16", [2000, 17], dict(D=256, Hkv=2, group=4, q_len=1, page_size=64)),
    ("bf16_d128", "bf16", [1500, 2048, 17], dict(Hkv=8, group=4, q_len=1)),
    ("bf16_d128_q4_8B", "bf16", [333, 1], dict(Hkv=2, group=4, q_len=4, layout="interleaved", base_pad=8)),
    # bases 8 bytes past a 16-byte boundary with 16-byte strides load through
    # TMA windows: pieces of 64 + 16 slots, whole in-page tiles, many splits
    ("fp8_page80_window", "fp8", [1000, 333], dict(Hkv=2, page_size=80, layout="interleaved", base_pad=8)),
    ("fp8_page208_window_splits", "fp8", [20000, 4097], dict(page_size=208, layout="interleaved", base_pad=8)),
    ("e5m2_page144_window", "e5m2", [900, 131], dict(Hkv=2, page_size=144, layout="interleaved", base_pad=8)),
    ("f16_page208_window", "f16", [3000, 129], dict(page_size=208, layout="interleaved", base_pad=8)),
    ("bf16_d256_page144_window", "bf16", [1500, 77],
     dict(D=256, Hkv=2, page_size=144, layout="interleaved", base_pad=8)),
    # token strides 8 past a multiple of 16: the cp.async loader
    ("fp8_padded_tokens_copy", "fp8", [700, 129, 0], dict(Hkv=2, page_size=32, layout="padded_tokens", base_pad=8)),
    ("e5m2_padded_tokens_copy", "e5m2", [300, 37], dict(layout="padded_tokens")),
    ("f16_padded_tokens_copy", "f16", [700, 129, 0], dict(Hkv=2, page_size=32, layout="padded_tokens")),
    ("bf16_d256_padded_tokens_copy", "bf16", [500, 33], dict(D=256, Hkv=2, layout="padded_tokens")),
    ("bf16_d128_padded_tokens_copy", "bf16", [333, 1], dict(Hkv=2, group=4, q_len=4, layout="padded_tokens")),
]


def _expected_load_path(kw):
    if kw.get("layout") == "padded_tokens":
        return B.PA_KV_LOAD_COPY
    return B.PA_KV_LOAD_WINDOW if kw.get("base_pad", 0) == 8 else B.PA_KV_LOAD_TMA


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_load_path_of_each_layout(case):
    """Each parity case runs the K/V load path its alignment calls for: the
    CUDA driver accepts every tensor map, so nothing falls back silently."""
    _, kind, lens, kw = case
    w = _small(kind, lens, **kw)
    kv = w.kv.data_ptr()
    st, path = B.pa_debug_kv_load_path(D.params_for(w), w.spec.head_dim, w.spec.elem_bytes, kv + w.k_offset,
                                       kv + w.v_offset)
    assert st == B.PA_OK
    assert path == _expected_load_path(kw)


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_against_oracle(case):
    _, kind, lens, kw = case
    w = _small(kind, lens, **kw)
    dec = D.Decoder(w, with_lse=(kind == "bf16"))
    dec.run()
    torch.cuda.synchronize()
    assert dec.status() == 0
    check_full(w, dec.out, dec.lse)


# ----------------------------------------------------------- full-size configs --

def _full(name, w_index=0):
    spec = wl.SPECS[name]
    return wl.generate(spec, wl.working_set_seed(name, w_index), device="cuda")


def test_config_b1_l3297():
    w = _full("b1_l3297")
    dec = D.Decoder(w)
    dec.run()
    torch.cuda.synchronize()
    assert dec.status() == 0
    check_full(w, dec.out)


def test_config_b4_l32k():
    w = _full("b4_l32k", 3)
    dec = D.Decoder(w)
    dec.run()
    torch.cuda.synchronize()
    assert dec.status() == 0
    check_full(w, dec.out)


def test_config_b1_l3297_e5m2():
    w = _full("b1_l3297_e5m2")
    dec = D.Decoder(w)
    dec.run()
    torch.cuda.synchronize()
    assert dec.status() == 0
    check_full(w, dec.out)


@pytest.mark.parametrize("name", ["b1_l3297_f16", "b1_l3297_bf16"])
def test_config_b1_l3297_16bit(name):
    w = _full(name)
    dec = D.Decoder(w, with_lse=w.spec.kind == "bf16")
    dec.run()
    torch.cuda.synchronize()
    assert dec.status() == 0
    check_full(w, dec.out, dec.lse)


def test_e4m3_every_finite_code():
    """K and V bytes drawn uniformly from all 254 finite E4M3 codes (both
    zeros, subnormals 2^-9 .. 7 * 2^-9, normals up to 448); 0x7F and 0xFF (NaN)
    are outside the contract and never drawn."""
    w = _small("fp8", [700, 260], page_size=32, seed=15)
    g = torch.Generator().manual_seed(16)
    kv = w.kv.cpu()
    n = w.v_offset - w.k_offset
    codes = torch.randint(0, 254, (2 * n,), generator=g, dtype=torch.int64)
    codes = codes + (codes >= 0x7F).long()  # 0..253 -> the 254 codes other than 0x7F and 0xFF
    kv[w.k_offset:w.k_offset + 2 * n] = codes.to(torch.uint8)
    assert set(kv[w.k_offset:w.k_offset + 2 * n].unique().tolist()) == set(range(256)) - {0x7F, 0xFF}
    w = wl.Workload(**{**w.__dict__, "kv": kv.cuda(), "k_scale": 1.0 / 448, "v_scale": 1.0 / 448})
    dec = D.Decoder(w)
    dec.run()
    torch.cuda.synchronize()
    assert dec.status() == 0
    check_full(w, dec.out)


def test_e5m2_every_finite_code():
    """K and V bytes drawn uniformly from all 248 finite E5M2 codes (subnormals,
    both zeros, 2^-16 .. 57344), so the decode is exercised on every code."""
    w = _small("e5m2", [700, 260], page_size=32, seed=13)
    g = torch.Generator().manual_seed(14)
    kv = w.kv.cpu()
    n = w.v_offset - w.k_offset
    codes = torch.randint(0, 256, (2 * n,), generator=g, dtype=torch.int64)
    finite = ((codes >> 2) & 31) != 31
    codes = torch.where(finite, codes, codes & 0x83)      # exponent 31 -> 0 (a subnormal)
    kv[w.k_offset:w.k_offset + 2 * n] = codes.to(torch.uint8)
    assert set(kv[w.k_offset:w.k_offset + 2 * n].unique().tolist()) == {c for c in range(256) if (c >> 2) & 31 != 31}
    w = wl.Workload(**{**w.__dict__, "kv": kv.cuda(), "k_scale": 2.0 / 57344, "v_scale": 1.0 / 57344})
    dec = D.Decoder(w)
    dec.run()
    torch.cuda.synchronize()
    assert dec.status() == 0
    check_full(w, dec.out)


def _sample_rows(w, per_request: int, seed: int) -> np.ndarray:
    s = w.spec
    rng = np.random.default_rng(seed)
    rows = []
    for b in range(s.batch):
        base = b * s.q_len * s.num_q_heads
        # always the first and last verify query of the first and last head, plus random ones
        fixed = [base, base + s.num_q_heads - 1, base + (s.q_len - 1) * s.num_q_heads,
                 base + s.q_len * s.num_q_heads - 1]
        rnd = rng.integers(0, s.q_len * s.num_q_heads, per_request) + base
        rows.extend(fixed + list(rnd))
    return np.unique(np.array(rows, dtype=np.int32))


def test_config_b8_l128k_every_row():
    """The benchmark workload (B8 x 131072 keys, E4M3) in the benchmark's
    launch configuration: all 384 output rows against the oracle."""
    w = _full("b8_l128k")
    dec = D.Decoder(w)
    dec.run()
    torch.cuda.synchronize()
    assert dec.status() == 0
    check_full(w, dec.out)


def test_config_b8_l128k_e5m2_sampled():
    w = _full("b8_l128k_e5m2")
    dec = D.Decoder(w)
    dec.run()
    torch.cuda.synchronize()
    assert dec.status() == 0
    check_rows(w, dec.out, _sample_rows(w, 2, 6))
    assert torch.isfinite(dec.out.float()).all()


@pytest.mark.parametrize("name", ["b8_l128k_f16", "b8_l128k_bf16"])
def test_config_b8_l128k_16bit_sampled(name):
    w = _full(name)
    dec = D.Decoder(w)
    dec.run()
    torch.cuda.synchronize()
    assert dec.status() == 0
    check_rows(w, dec.out, _sample_rows(w, 2, 7))
    assert torch.isfinite(dec.out.float()).all()


def test_config_b16_mixed_sampled():
    w = _full("b16_mixed")
    kv = w.kv.data_ptr()
    # 8-byte-only aligned bases with 16-byte strides: TMA windows
    assert B.pa_debug_kv_load_path(D.params_for(w), 256, 1, kv + w.k_offset, kv + w.v_offset) == \
        (B.PA_OK, B.PA_KV_LOAD_WINDOW)
    dec = D.Decoder(w)
    dec.run()
    torch.cuda.synchronize()
    assert dec.status() == 0
    out = dec.out
    lens = w.ctx_lens.cpu().tolist()
    for b, L in enumerate(lens):
        if L == 0:
            assert torch.all(out[b] == 0) and not torch.signbit(out[b].float()).any()
    # the longest and the shortest live request in full, the rest sampled
    live = [b for b, L in enumerate(lens) if L > 0]
    longest, shortest = max(live, key=lambda b: lens[b]), min(live, key=lambda b: lens[b])
    s = w.spec
    per = s.q_len * s.num_q_heads
    rows = set(range(longest * per, (longest + 1) * per)) | set(range(shortest * per, (shortest + 1) * per))
    rows |= set(_sample_rows(w, 1, 9).tolist())
    check_rows(w, out, np.array(sorted(rows), dtype=np.int32))


@pytest.mark.parametrize("b", [1, 2, 4, 8])
def test_config_d128(b):
    w = _full(f"d128_b{b}")
    dec = D.Decoder(w, with_lse=True)
    dec.run()
    torch.cuda.synchronize()
    assert dec.status() == 0
    check_full(w, dec.out, dec.lse)


# ------------------------------------------------------------ invariants --

def _single(w, b):
    """Request b of workload w as a batch of one (same KV buffer and pool)."""
    s = w.spec
    spec1 = wl.Spec(s.name + "_single", s.kind, 1, s.num_kv_heads, s.num_q_heads, s.head_dim, s.q_len,
                    s.page_size, s.max_ctx_len, ctx_lens=(0,), layout=s.layout, base_pad=s.base_pad)
    return wl.Workload(spec=spec1, q=w.q[b:b + 1].clone(), kv=w.kv, k_offset=w.k_offset, v_offset=w.v_offset,
                       k_strides=w.k_strides, v_strides=w.v_strides, block_table=w.block_table[b:b + 1].clone(),
                       ctx_lens=w.ctx_lens[b:b + 1].clone(), num_pages=w.num_pages, k_scale=w.k_scale,
                       v_scale=w.v_scale)


@pytest.mark.parametrize("name", ["b8_l128k", "b4_l32k", "b16_mixed", "d128_b8", "b8_l128k_e5m2", "b8_l128k_f16"])
def test_batched_equals_single_bitwise(name):
    w = _full(name)
    batched = D.Decoder(w).run().clone()
    for b in range(w.spec.batch):
        one = D.Decoder(_single(w, b)).run()
        assert torch.equal(one[0].view(torch.int16), batched[b].view(torch.int16)), f"request {b} differs"


@pytest.mark.parametrize("name", ["b16_mixed", "b8_l128k", "b8_l128k_f16"])
def test_repeated_calls_bitwise_equal(name):
    """Repeated calls on the same inputs give the same bits.  The staging tiles
    are read by the decode warps through the generic proxy and refilled by TMA
    through the async proxy; a missing order between the two showed as
    call-to-call differences on the 8-byte aligned (window) layout, whose K and
    V rows share L2 lines and so land soonest after a release."""
    w = _full(name)
    dec = D.Decoder(w)
    first = dec.run().clone()
    for _ in range(4):
        again = dec.run()
        torch.cuda.synchronize()
        assert dec.status() == 0
        assert torch.equal(first.view(torch.int16), again.view(torch.int16))


def test_graph_replay_with_changed_inputs():
    w = _full("b4_l32k", 1)
    dec = D.Decoder(w)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        B.check(dec(s), "warm-up")
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        B.check(dec(torch.cuda.current_stream()), "captured call")
    g.replay()
    torch.cuda.synchronize()
    ref1 = D.Decoder(w).run().clone()
    assert torch.equal(dec.out.view(torch.int16), ref1.view(torch.int16))
    # change Q, lengths (including a zero row) and scales in place, replay
    w.q.copy_(torch.randn_like(w.q.float()).half())
    w.ctx_lens.copy_(torch.tensor([32768, 77, 0, 20001], dtype=torch.int32))
    dec.scales.mul_(1.5)
    g.replay()
    torch.cuda.synchronize()
    w2 = wl.Workload(**{**w.__dict__, "k_scale": float(dec.scales[0]), "v_scale": float(dec.scales[1])})
    ref2 = D.Decoder(w2).run().clone()
    assert torch.equal(dec.out.view(torch.int16), ref2.view(torch.int16))
    check_full(w2, dec.out)


# ---------------------------------------------------------- bookkeeping --

def schedule(lens, Hkv):
    """Restatement of the persistent schedule: requests by split length
    descending (ties by index), then KV head, then split."""
    plans = []
    for L in lens:
        st, s, c = B.pa_split_plan(max(L, 0), Hkv)
        plans.append((s, c))
    order = sorted(range(len(lens)), key=lambda b: (-plans[b][1], b))
    items = []
    for b in order:
        s, c = plans[b]
        for g in range(Hkv):
            for k in range(s):
                items.append((b, g, k * c, min((k + 1) * c, lens[b])))
    return items


def test_worklist_bit_exact():
    lens = [131072, 0, 3297, 262144, 1, 129, 77777, 0, 8]
    spec = wl.Spec("wl", "fp8", len(lens), 2, 12, 256, 8, 3296, 262144, ctx_lens=tuple(lens))
    w = wl.generate(spec, 3)
    p = D.params_for(w)
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    cap = len(lens) * 2 * B.pa_get_capabilities().max_splits
    items = torch.full((cap, 4), -7, dtype=torch.int32, device="cuda")
    count = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.check(B.pa_debug_worklist(p, cl, items, cap, count), "pa_debug_worklist")
    torch.cuda.synchronize()
    want = schedule(lens, 2)
    assert int(count) == len(want)
    assert [tuple(r) for r in items[:len(want)].cpu().tolist()] == want


@pytest.mark.parametrize("layout,pad", [("separate", 0), ("interleaved", 8)])
def test_gather_bit_exact(layout, pad):
    lens = [3297, 1, 0, 2000]
    spec = wl.Spec("ga", "fp8", len(lens), 2, 12, 256, 8, 1648, 4000, ctx_lens=tuple(lens), layout=layout,
                   base_pad=pad)
    w = wl.generate(spec, 4).to("cuda")
    p = D.params_for(w)
    kv = w.kv.data_ptr()
    for which, off, st in ((0, w.k_offset, w.k_strides), (1, w.v_offset, w.v_strides)):
        dst = torch.zeros((len(lens), 2, spec.max_ctx_len, 256), dtype=torch.uint8, device="cuda")
        B.check(B.pa_debug_gather_fp8(p, kv + w.k_offset, kv + w.v_offset, w.block_table, w.ctx_lens, which, dst),
                "gather")
        torch.cuda.synchronize()
        host = w.kv.cpu().numpy()
        bt = w.block_table.cpu().numpy()
        got = dst.cpu().numpy()
        for b, L in enumerate(lens):
            for g in range(2):
                want = np.stack([host[off + bt[b, j // 1648] * st[0] + (j % 1648) * st[1] + g * st[2]:][:256]
                                 for j in range(L)]) if L else np.zeros((0, 256), np.uint8)
                assert np.array_equal(got[b, g, :L], want)


def test_all_zero_batch_writes_zeros():
    """Every request of the batch has length 0 (an all-padding batch): no work
    item exists, every output element is +0.0, LSE is -inf and no flag is set;
    then the same decoder serves live lengths again."""
    for kind, kw in (("fp8", {}), ("f16", {}), ("bf16", dict(D=256)), ("bf16", dict(Hkv=8, group=4, q_len=1))):
        w = _small(kind, [0, 0, 0], max_ctx=4000, **kw)
        w.q.fill_(float("nan"))
        dec = D.Decoder(w, with_lse=(kind == "bf16"))
        dec.out.fill_(7.0)
        dec.run()
        torch.cuda.synchronize()
        assert dec.status() == 0
        assert torch.all(dec.out == 0) and not torch.signbit(dec.out.float()).any(), kind
        if dec.lse is not None:
            assert torch.all(dec.lse == float("-inf"))
    w = _small("fp8", [0, 500, 0], max_ctx=4000, seed=3)
    dec = D.Decoder(w)
    w.ctx_lens.zero_()
    dec.run()
    torch.cuda.synchronize()
    assert dec.status() == 0 and torch.all(dec.out == 0)
    w.ctx_lens.copy_(torch.tensor([0, 500, 0], dtype=torch.int32))
    dec.run()
    torch.cuda.synchronize()
    assert dec.status() == 0
    check_full(w, dec.out)


# ------------------------------------------------------------ input checks --

def test_bad_page_flags_and_zeros_request():
    w = _small("fp8", [400, 300, 50], page_size=32, seed=7)
    w.block_table[1, 3] = w.num_pages + 5
    dec = D.Decoder(w)
    dec.run()
    torch.cuda.synchronize()
    assert dec.status() & B.PA_FLAG_BAD_PAGE
    assert torch.all(dec.out[1] == 0)
    from helpers import run_oracle
    ref, _ = run_oracle(w.to("cpu").__class__(**{**w.to("cpu").__dict__}), rows=np.arange(0, 48, dtype=np.int32))
    assert np.abs(to_f64(dec.out[0]).reshape(48, 256) - ref).max() <= 2e-3
    B.check(B.pa_clear_status(dec.workspace), "clear")
    assert dec.status() == 0


def test_bad_length_flags_and_zeros_request():
    w = _small("fp8", [400, 300], page_size=32, seed=8, max_ctx=512)
    w.ctx_lens[0] = 513  # beyond max_ctx_len
    dec = D.Decoder(w)
    dec.run()
    torch.cuda.synchronize()
    assert dec.status() & B.PA_FLAG_BAD_LENGTH
    assert torch.all(dec.out[0] == 0)
    w.ctx_lens[0] = -3
    B.check(B.pa_clear_status(dec.workspace), "clear")
    dec.run()
    torch.cuda.synchronize()
    assert dec.status() & B.PA_FLAG_BAD_LENGTH
    assert torch.all(dec.out[0] == 0)


# ------------------------------------------------------ online-softmax rescale --

def test_growing_scores_force_rescales():
    """Scores that grow along the context move each row's running maximum by
    far more than the lazy threshold many times (the O^T rescale path)."""
    lens = [2000, 700]
    w = _small("fp8", lens, page_size=16, seed=11)
    s = w.spec
    w.q.fill_(1.0)
    # K row of key j: every element the E4M3 code of a value growing with j
    codes = torch.tensor([0x20 + (j * 0x5B) // 2000 for j in range(max(lens))], dtype=torch.uint8)
    kv = w.kv.cpu()
    bt = w.block_table.cpu()
    for b, L in enumerate(lens):
        for j in range(L):
            page = int(bt[b, j // s.page_size])
            start = w.k_offset + page * w.k_strides[0] + (j % s.page_size) * w.k_strides[1]
            kv[start:start + 256] = codes[j]
    w = wl.Workload(**{**w.__dict__, "kv": kv.cuda(), "k_scale": 0.02})
    dec = D.Decoder(w)
    dec.run()
    torch.cuda.synchronize()
    assert dec.status() == 0
    check_full(w, dec.out)


# ------------------------------------------------------------ bounded waits --

def test_wait_bound_runs_out_cleanly():
    """With the Q-ready signal withheld and a ~10 ms wait bound, every CTA must
    give up, free its tensor memory and raise PA_FLAG_TIMEOUT; the context
    stays usable and the next call is correct."""
    import time

    w = _small("fp8", [3000, 700, 37], seed=21)
    dec = D.Decoder(w)
    B.check(B.pa_debug_stall_next(20_000_000), "pa_debug_stall_next")
    t0 = time.perf_counter()
    B.check(dec(), "stalled call")
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 30.0
    assert dec.status() & B.PA_FLAG_TIMEOUT
    B.check(B.pa_clear_status(dec.workspace), "clear")
    dec.run()
    torch.cuda.synchronize()
    assert dec.status() == 0
    check_full(w, dec.out)
    assert B.pa_debug_stall_next(0) == B.PA_ERR_SHAPE


def test_per_call_words_return_to_zero():
    """A decode call leaves its per-request flags, arrival counters and task
    counters at zero (the last CTA resets them), also after a call that saw
    a bad length, so the next call on the same workspace needs no clearing."""
    w = _small("fp8", [3000, 700, 37], seed=23)
    dec = D.Decoder(w)
    good = w.ctx_lens.clone()
    for lens in (good, torch.tensor([3000, 10**9, 37], dtype=torch.int32, device="cuda"), good):
        w.ctx_lens.copy_(lens)
        dec.run()
        torch.cuda.synchronize()
        words = dec.workspace[512:1032].view(torch.int32)
        assert torch.count_nonzero(words) == 0
    B.check(B.pa_clear_status(dec.workspace), "clear")
    dec.run()
    torch.cuda.synchronize()
    assert dec.status() == 0
    check_full(w, dec.out)
