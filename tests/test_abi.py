"""The C-ABI library on the host (no GPU needed): it loads, exports every entry
point include/pa.h declares, reports its capabilities, plans splits as the
restatement below does, sizes workspaces, and rejects every bad argument
before touching CUDA."""
import ctypes
import math

import pytest

from paged_gqa_decode_split_gb300 import binding as B
from paged_gqa_decode_split_gb300 import build as pa_build


@pytest.fixture(scope="module")
def lib():
    pa_build.build()
    return B.load()


def test_exports_every_declared_symbol(lib):
    names = B.header_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), f"{n} declared in pa.h but not exported"


def test_capabilities(lib):
    c = B.pa_get_capabilities()
    assert c.abi_version == 2
    assert c.accum_bits == 32
    assert c.page_multiple == 16
    assert c.fp8_head_dim == 256 and c.bf16_head_dim == 128
    assert c.max_splits == 38 and all(r == 0 for r in c.reserved)
    assert c.max_q_len >= 8 and c.max_group >= 6 and c.max_batch >= 16 and c.max_ctx >= 262144
    assert lib.pa_get_capabilities(None) == B.PA_ERR_NULL


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6, 42):
        assert isinstance(B.status_string(code), str) and B.status_string(code)


def splits_for_len(L: int, hkv: int = 1) -> tuple[int, int]:
    """Restatement of the split policy: about 512 * min(Hkv, 4) keys per
    split, at most 38 splits (a quarter of the 152 SMs), split length a whole
    number of 128-key tiles."""
    if L <= 0:
        return 0, 0
    s0 = min(max(math.ceil(L / (512 * min(hkv, 4))), 1), 38)
    chunk = math.ceil(math.ceil(L / s0) / 128) * 128
    return math.ceil(L / chunk), chunk


@pytest.mark.parametrize("hkv", [1, 2, 3, 8])
@pytest.mark.parametrize("L", [0, 1, 7, 8, 127, 128, 129, 511, 512, 513, 3297, 16383, 32768, 131072, 131073,
                               200000, 262144, 1 << 20])
def test_split_plan_matches_restatement(lib, L, hkv):
    st, s, c = B.pa_split_plan(L, hkv)
    assert st == 0
    assert (s, c) == splits_for_len(L, hkv)
    if L > 0:
        assert 1 <= s <= 38 and c % 128 == 0
        assert (s - 1) * c < L <= s * c  # every split non-empty


def test_split_count_bounded_by_workspace_bound(lib):
    """The count is not monotone in L (S(19456) = 38, S(19457) = 31), so the
    workspace is sized with the monotone bound clamp(ceil(max_ctx/512), 1, 38);
    no length up to max_ctx may need more splits than that."""
    assert B.pa_split_plan(19456)[1] == 38 and B.pa_split_plan(19457)[1] == 31
    worst = 0
    for L in range(0, 70000, 7):
        worst = max(worst, B.pa_split_plan(L)[1])
        for hkv in (1, 2, 4, 8):
            assert B.pa_split_plan(L, hkv)[1] <= min(38, max(1, math.ceil(L / 512)))
    assert worst == 38
    # the workspace of max_ctx_len 19457 must hold 38 splits per (request, KV head)
    p = _params(max_ctx_len=19457, max_pages_per_req=12)
    assert B.pa_decode_fp8_workspace_bytes(p) >= 1024 + 8 * 38 * 48 * (256 * 4 + 8)


def test_split_plan_rejects_negative(lib):
    assert B.pa_split_plan(-1)[0] == B.PA_ERR_SHAPE
    assert B.pa_split_plan(100, 0)[0] == B.PA_ERR_SHAPE


def test_split_plan_known_configs(lib):
    assert B.pa_split_plan(131072)[1:] == (38, 3456)
    assert B.pa_split_plan(32768)[1:] == (37, 896)
    assert B.pa_split_plan(3297)[1:] == (7, 512)
    assert B.pa_split_plan(262144)[1:] == (38, 6912)
    # the head count stretches the split floor: 8 KV heads give splits of 2048 keys or more
    assert B.pa_split_plan(16384, 8)[1:] == (8, 2048)
    assert B.pa_split_plan(262144, 2)[1:] == (38, 6912)


def _params(**kw):
    base = dict(batch=8, num_kv_heads=1, num_q_heads=6, head_dim=256, q_len=8, page_size=1648,
                max_pages_per_req=80, num_pages=640, max_ctx_len=131072, k_strides=(1648 * 256, 256, 256),
                v_strides=(1648 * 256, 256, 256))
    base.update(kw)
    return B.make_params(**base)


def test_workspace_size_formula(lib):
    p = _params()
    n = B.pa_decode_fp8_workspace_bytes(p)
    items = 8 * 1 * 38 * 48
    assert n >= 1024 + items * 8 + items * 256 * 4
    assert n % 256 == 0
    assert B.pa_decode_fp8_workspace_bytes(_params(head_dim=128)) == 0
    q = _params(head_dim=128, num_kv_heads=8, num_q_heads=32, q_len=1, page_size=16, max_pages_per_req=2048,
                max_ctx_len=32768, k_strides=(16 * 8 * 256, 8 * 256, 256), v_strides=(16 * 8 * 256, 8 * 256, 256))
    assert B.pa_decode_bf16_d128_workspace_bytes(q) >= 1024 + 8 * 8 * 32 * 4 * (128 * 4 + 8)


FAKE = 0x10000  # 64 KiB-aligned fake device address: never dereferenced, every check fails first


def _call(p, **over):
    args = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, cl=FAKE, ks=FAKE, vs=FAKE, out=FAKE, ws=FAKE,
                ws_bytes=1 << 40)
    args.update(over)
    return B.pa_decode_fp8(p, args["q"], args["k"], args["v"], args["bt"], args["cl"], args["ks"], args["vs"],
                           args["out"], args["ws"], args["ws_bytes"], 0)


@pytest.mark.parametrize("over,expect", [
    (dict(head_dim=128), B.PA_ERR_UNSUPPORTED),
    (dict(batch=0), B.PA_ERR_SHAPE),
    (dict(batch=65), B.PA_ERR_SHAPE),
    (dict(q_len=0), B.PA_ERR_SHAPE),
    (dict(q_len=9), B.PA_ERR_SHAPE),
    (dict(num_kv_heads=2, num_q_heads=7), B.PA_ERR_SHAPE),   # heads not a multiple of KV heads
    (dict(num_kv_heads=0), B.PA_ERR_SHAPE),
    (dict(num_q_heads=18), B.PA_ERR_UNSUPPORTED),            # GQA 18 > max_group
    (dict(page_size=1000), B.PA_ERR_SHAPE),
    (dict(page_size=0), B.PA_ERR_SHAPE),
    (dict(max_pages_per_req=10), B.PA_ERR_SHAPE),
    (dict(max_ctx_len=-1), B.PA_ERR_SHAPE),
    (dict(max_ctx_len=(1 << 20) + 1, max_pages_per_req=1 << 20), B.PA_ERR_SHAPE),
    (dict(num_pages=0), B.PA_ERR_SHAPE),
], ids=lambda x: str(x))
def test_rejects_bad_geometry(lib, over, expect):
    assert _call(_params(**over)) == expect


def test_rejects_misaligned_strides(lib):
    assert _call(_params(k_strides=(1648 * 256, 260, 256))) == B.PA_ERR_ALIGN
    assert _call(_params(v_strides=(1648 * 256, 256, -256))) == B.PA_ERR_SHAPE


@pytest.mark.parametrize("arg", ["q", "k", "v", "bt", "cl", "ks", "vs", "out"])
def test_rejects_null_pointers(lib, arg):
    assert _call(_params(), **{arg: 0}) == B.PA_ERR_NULL


def test_rejects_misaligned_pointers(lib):
    assert _call(_params(), q=FAKE + 8) == B.PA_ERR_ALIGN
    assert _call(_params(), out=FAKE + 2) == B.PA_ERR_ALIGN
    assert _call(_params(), k=FAKE + 4) == B.PA_ERR_ALIGN


def test_rejects_bad_workspace(lib):
    p = _params()
    need = B.pa_decode_fp8_workspace_bytes(p)
    assert _call(p, ws=0) == B.PA_ERR_WORKSPACE
    assert _call(p, ws=FAKE + 128) == B.PA_ERR_WORKSPACE
    assert _call(p, ws_bytes=need - 1) == B.PA_ERR_WORKSPACE


def test_null_params(lib):
    assert lib.pa_decode_fp8(None, *([ctypes.c_void_p(FAKE)] * 9), 1 << 30, None) == B.PA_ERR_NULL
    assert lib.pa_decode_fp8_workspace_bytes(None) == 0


def test_e5m2_entry_validates(lib):
    """pa_decode_e5m2 runs the same host checks as pa_decode_fp8 before any launch."""
    p = _params()
    ok = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, cl=FAKE, ks=FAKE, vs=FAKE, out=FAKE, ws=FAKE, n=1 << 40)

    def call(params=p, **o):
        a = {**ok, **o}
        return B.pa_decode_e5m2(params, a["q"], a["k"], a["v"], a["bt"], a["cl"], a["ks"], a["vs"], a["out"],
                                a["ws"], a["n"], 0)
    for arg in ("q", "k", "v", "bt", "cl", "ks", "vs", "out"):
        assert call(**{arg: 0}) == B.PA_ERR_NULL, arg
    assert call(q=FAKE + 8) == B.PA_ERR_ALIGN
    assert call(ks=FAKE + 2) == B.PA_ERR_ALIGN
    assert call(ws=0) == B.PA_ERR_WORKSPACE
    assert call(n=B.pa_decode_fp8_workspace_bytes(p) - 1) == B.PA_ERR_WORKSPACE
    assert call(params=_params(head_dim=128)) == B.PA_ERR_UNSUPPORTED
    assert call(params=_params(q_len=9)) == B.PA_ERR_SHAPE
    assert lib.pa_decode_e5m2(None, *([ctypes.c_void_p(FAKE)] * 9), 1 << 30, None) == B.PA_ERR_NULL


def test_16bit_d256_entries_validate(lib):
    """pa_decode_f16 and pa_decode_bf16_d256 take no scales and run the D 256 checks."""
    p = _params()
    ok = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, cl=FAKE, out=FAKE, lse=None, ws=FAKE, n=1 << 40)

    def f16(params=p, **o):
        a = {**ok, **o}
        return B.pa_decode_f16(params, a["q"], a["k"], a["v"], a["bt"], a["cl"], a["out"], a["ws"], a["n"], 0)

    def bf16(params=p, **o):
        a = {**ok, **o}
        return B.pa_decode_bf16_d256(params, a["q"], a["k"], a["v"], a["bt"], a["cl"], a["out"], a["lse"], a["ws"],
                                     a["n"], 0)
    for call in (f16, bf16):
        for arg in ("q", "k", "v", "bt", "cl", "out"):
            assert call(**{arg: 0}) == B.PA_ERR_NULL, arg
        assert call(q=FAKE + 8) == B.PA_ERR_ALIGN
        assert call(k=FAKE + 4) == B.PA_ERR_ALIGN
        assert call(ws=0) == B.PA_ERR_WORKSPACE
        assert call(n=B.pa_decode_fp8_workspace_bytes(p) - 1) == B.PA_ERR_WORKSPACE
        assert call(params=_params(head_dim=128)) == B.PA_ERR_UNSUPPORTED
        assert call(params=_params(batch=0)) == B.PA_ERR_SHAPE
    assert bf16(lse=FAKE + 4) == B.PA_ERR_ALIGN
    assert lib.pa_decode_f16(None, *([ctypes.c_void_p(FAKE)] * 7), 1 << 30, None) == B.PA_ERR_NULL


def test_bf16_entry_validates(lib):
    p = _params(head_dim=128, num_kv_heads=8, num_q_heads=32, q_len=1, page_size=16, max_pages_per_req=2048,
                max_ctx_len=32768, k_strides=(16 * 8 * 256, 8 * 256, 256), v_strides=(16 * 8 * 256, 8 * 256, 256))
    ok = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, cl=FAKE, out=FAKE, lse=None, ws=FAKE, n=1 << 40)

    def call(**o):
        a = {**ok, **o}
        return B.pa_decode_bf16_d128(p, a["q"], a["k"], a["v"], a["bt"], a["cl"], a["out"], a["lse"], a["ws"],
                                     a["n"], 0)
    assert call(q=0) == B.PA_ERR_NULL
    assert call(lse=FAKE + 4) == B.PA_ERR_ALIGN
    assert call(n=0) == B.PA_ERR_WORKSPACE
    p.head_dim = 256
    assert call() == B.PA_ERR_UNSUPPORTED


def test_timing_and_status_arguments(lib):
    assert B.pa_timing_enable(False) == 0
    assert B.pa_timing_collect(2)[0] == B.PA_ERR_SHAPE
    st, ms, n = B.pa_timing_collect(0)
    assert st == 0 and n == 0 and ms == 0.0
    assert lib.pa_read_status(None, None, None) == B.PA_ERR_NULL
    assert lib.pa_clear_status(None, None) == B.PA_ERR_NULL


# ------------------------------------------------------------------ prefill --

def _prefill_params(**over):
    p = B.pa_prefill_params()
    p.batch, p.q_len, p.kv_len, p.num_q_heads, p.num_kv_heads, p.head_dim = 2, 300, 5000, 12, 2, 256
    ts = 2 * 256 + 8
    p.k_batch_stride, p.k_token_stride, p.k_head_stride = 5000 * ts, ts, 256
    p.v_batch_stride, p.v_token_stride, p.v_head_stride = 5000 * ts, ts, 256
    for k, v in over.items():
        setattr(p, k, v)
    return p


def _prefill_plan_restated(kv):
    """split_len 32768 above 32768 keys, else ceil(kv / 8) rounded up to 128, at least 1024."""
    ln = 32768 if kv > 32768 else max(1024, -(-(-(-kv // 8)) // 128) * 128)
    return -(-kv // ln), ln


@pytest.mark.parametrize("kv", [1, 100, 1024, 1025, 8192, 8193, 20000, 32768, 32769, 70000, 262144, 1 << 22])
def test_prefill_plan_matches_statement(lib, kv):
    st, ns, ln = B.pa_prefill_plan(kv)
    assert st == B.PA_OK and (ns, ln) == _prefill_plan_restated(kv)
    assert ln % 128 == 0 and (ns - 1) * ln < kv <= ns * ln


def test_prefill_plan_known_values(lib):
    assert B.pa_prefill_plan(262144)[1:] == (8, 32768)
    assert B.pa_prefill_plan(5000)[1:] == (5, 1024)
    assert B.pa_prefill_plan(0)[0] == B.PA_ERR_SHAPE
    assert lib.pa_prefill_plan(10, None, None) == B.PA_ERR_NULL


def test_prefill_workspace_size_formula(lib):
    p = _prefill_params()
    ns, _ = _prefill_plan_restated(p.kv_len)
    tiles = p.batch * p.num_q_heads * math.ceil(p.q_len / 128) * ns
    rows = tiles * 128
    ml = (rows * 8 + 255) // 256 * 256
    assert B.pa_prefill_f16_workspace_bytes(p) == 256 + ml + rows * 256 * 4
    # the headline shape: 8 splits x 64 query tiles x 6 heads
    big = _prefill_params(batch=1, q_len=8192, kv_len=262144, num_q_heads=6, num_kv_heads=1)
    assert B.pa_prefill_f16_workspace_bytes(big) == 256 + 384 * 8 * 128 * 8 + 384 * 8 * 128 * 1024


@pytest.mark.parametrize("over", [dict(head_dim=128), dict(batch=0), dict(batch=65), dict(q_len=0),
                                  dict(kv_len=0), dict(num_kv_heads=5), dict(num_q_heads=0),
                                  dict(k_token_stride=516), dict(v_head_stride=-256), dict(k_batch_stride=0)])
def test_prefill_rejects_bad_geometry(lib, over):
    p = _prefill_params(**over)
    assert B.pa_prefill_f16_workspace_bytes(p) == 0
    st = B.pa_prefill_f16(p, 256, 512, 768, 1024, None, 4096, 1 << 30, stream=0)
    assert st in (B.PA_ERR_SHAPE, B.PA_ERR_UNSUPPORTED, B.PA_ERR_ALIGN)
    if "head_dim" in over:
        assert st == B.PA_ERR_UNSUPPORTED
    if "k_token_stride" in over:
        assert st == B.PA_ERR_ALIGN


def test_prefill_unit_extents_take_any_stride(lib):
    # batch 1 and one KV head: those strides are never applied
    p = _prefill_params(batch=1, num_kv_heads=1, num_q_heads=6, k_batch_stride=0, v_batch_stride=3,
                        k_head_stride=-1, v_head_stride=0)
    assert B.pa_prefill_f16_workspace_bytes(p) > 0


def test_prefill_rejects_bad_pointers_and_workspace(lib):
    p = _prefill_params()
    ws = B.pa_prefill_f16_workspace_bytes(p)
    assert lib.pa_prefill_f16(None, 256, 512, 768, 1024, None, 4096, ws, None) == B.PA_ERR_NULL
    assert B.pa_prefill_f16(p, None, 512, 768, 1024, None, 4096, ws, stream=0) == B.PA_ERR_NULL
    assert B.pa_prefill_f16(p, 256, 512, 768, None, None, 4096, ws, stream=0) == B.PA_ERR_NULL
    assert B.pa_prefill_f16(p, 264, 512, 768, 1024, None, 4096, ws, stream=0) == B.PA_ERR_ALIGN
    assert B.pa_prefill_f16(p, 256, 520, 768, 1024, None, 4096, ws, stream=0) == B.PA_ERR_ALIGN
    assert B.pa_prefill_f16(p, 256, 512, 768, 1032, None, 4096, ws, stream=0) == B.PA_ERR_ALIGN
    assert B.pa_prefill_f16(p, 256, 512, 768, 1024, 1026, 4096, ws, stream=0) == B.PA_ERR_ALIGN
    assert B.pa_prefill_f16(p, 256, 512, 768, 1024, None, 4096, ws - 1, stream=0) == B.PA_ERR_WORKSPACE
    assert B.pa_prefill_f16(p, 256, 512, 768, 1024, None, 4104, ws, stream=0) == B.PA_ERR_WORKSPACE
    assert B.pa_prefill_f16(p, 256, 512, 768, 1024, None, None, ws, stream=0) == B.PA_ERR_WORKSPACE
