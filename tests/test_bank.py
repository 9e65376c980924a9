"""Workspace bank (pa_bank_*) on the CPU: the bank makes no CUDA call, so a
fake allocator that hands out aligned fake addresses exercises every rule.

Rules ("DFlash2 concurrent long-context attention", sections "Why the
single-request optimization was missing from concurrent decode" and "Operator
validation"): one panel per (device, stream, context contract) shared by
every batch size it fits; descending sizes allocate once; growing allocates a
larger panel and keeps every older one (and every handed-out pointer) alive
until the bank is destroyed; different streams never share a panel."""
from __future__ import annotations

import threading

import pytest

from paged_gqa_decode_split_gb300 import binding as B


def _params(batch=8, **over):
    kw = dict(batch=batch, num_kv_heads=1, num_q_heads=6, head_dim=256, q_len=8, page_size=1648,
              max_pages_per_req=80, num_pages=640, max_ctx_len=131072,
              k_strides=(1648 * 256, 256, 256), v_strides=(1648 * 256, 256, 256))
    kw.update(over)
    return B.make_params(**kw)


class FakeDevice:
    """Hands out fake 256-byte aligned addresses; records every call."""

    def __init__(self, misalign=False, fail=False):
        self.next = 0x7000_0000_0000
        self.allocs, self.frees = [], []
        self.misalign, self.fail = misalign, fail
        self.lock = threading.Lock()

    def alloc(self, n, dev):
        with self.lock:
            if self.fail:
                return 0
            ptr = self.next + (8 if self.misalign else 0)
            self.next += (n + 4095) // 4096 * 4096 + 4096
            self.allocs.append((ptr, n, dev))
            return ptr

    def free(self, ptr, n, dev):
        with self.lock:
            self.frees.append((ptr, n, dev))


@pytest.fixture
def bank():
    B.load()
    fake = FakeDevice()
    h, keep = B.pa_bank_create(fake.alloc, fake.free)
    assert h
    yield h, fake
    assert B.pa_bank_destroy(h) == B.PA_OK


def _get(h, p, dev=0, stream=1):
    st, ptr, n = B.pa_bank_workspace(h, p, dev, stream)
    assert st == B.PA_OK, st
    return ptr, n


def test_descending_batches_allocate_once(bank):
    h, fake = bank
    ptrs = [_get(h, _params(batch=b))[0] for b in (16, 8, 4, 2, 1)]
    assert len(set(ptrs)) == 1 and len(fake.allocs) == 1
    assert fake.allocs[0][1] == B.pa_decode_fp8_workspace_bytes(_params(batch=16))
    assert B.pa_bank_stats(h)[1] == 1


def test_growing_keeps_older_panels(bank):
    h, fake = bank
    p2, n2 = _get(h, _params(batch=2))
    p8, n8 = _get(h, _params(batch=8))
    p16, n16 = _get(h, _params(batch=16))
    assert len({p2, p8, p16}) == 3 and n2 < n8 < n16
    # every later request of the key gets the largest panel; nothing was freed
    assert _get(h, _params(batch=2))[0] == p16
    assert _get(h, _params(batch=12))[0] == p16
    assert fake.frees == []
    st, panels, nbytes = B.pa_bank_stats(h)
    assert (st, panels, nbytes) == (B.PA_OK, 3, n2 + n8 + n16)


def test_keys_separate_streams_devices_and_contracts(bank):
    h, fake = bank
    base = _get(h, _params(batch=4))[0]
    assert _get(h, _params(batch=4), stream=2)[0] != base          # another stream
    assert _get(h, _params(batch=4), dev=1)[0] != base             # another device
    assert _get(h, _params(batch=4, q_len=4))[0] != base           # another verify window
    assert _get(h, _params(batch=4, max_ctx_len=32768, max_pages_per_req=20))[0] != base
    assert _get(h, _params(batch=4, num_kv_heads=2, num_q_heads=12))[0] != base
    # page size and strides are not part of the contract: the panel is shared
    assert _get(h, _params(batch=4, page_size=3296, max_pages_per_req=40,
                           k_strides=(3296 * 256, 256, 256), v_strides=(3296 * 256, 256, 256)))[0] == base
    assert len(fake.allocs) == 6


def test_bf16_contract(bank):
    h, fake = bank
    p = _params(batch=4, head_dim=128, num_kv_heads=8, num_q_heads=32, q_len=1, page_size=16,
                max_pages_per_req=2048, max_ctx_len=32768, k_strides=(16 * 8 * 256, 8 * 256, 256),
                v_strides=(16 * 8 * 256, 8 * 256, 256))
    ptr, n = _get(h, p)
    assert n == B.pa_decode_bf16_d128_workspace_bytes(p)


def test_destroy_releases_every_panel_once():
    B.load()
    fake = FakeDevice()
    h, keep = B.pa_bank_create(fake.alloc, fake.free)
    for b in (1, 4, 16):
        _get(h, _params(batch=b))
    _get(h, _params(batch=4), stream=9)
    assert B.pa_bank_destroy(h) == B.PA_OK
    assert sorted(fake.frees) == sorted(fake.allocs)


def test_errors():
    B.load()
    fake = FakeDevice(fail=True)
    h, keep = B.pa_bank_create(fake.alloc, fake.free)
    assert B.pa_bank_workspace(h, _params(), 0, 1)[0] == B.PA_ERR_WORKSPACE
    assert B.pa_bank_workspace(h, _params(head_dim=64), 0, 1)[0] == B.PA_ERR_UNSUPPORTED
    assert B.pa_bank_workspace(h, _params(q_len=9), 0, 1)[0] == B.PA_ERR_SHAPE
    assert B.pa_bank_workspace(h, _params(), -1, 1)[0] == B.PA_ERR_SHAPE
    assert fake.allocs == []
    assert B.pa_bank_stats(h)[1:] == (0, 0)
    assert B.pa_bank_destroy(h) == B.PA_OK
    # memory that is not 256-byte aligned is handed back and refused
    bad = FakeDevice(misalign=True)
    h, keep = B.pa_bank_create(bad.alloc, bad.free)
    assert B.pa_bank_workspace(h, _params(), 0, 1)[0] == B.PA_ERR_ALIGN
    assert bad.frees == bad.allocs and B.pa_bank_stats(h)[1] == 0
    assert B.pa_bank_destroy(h) == B.PA_OK
    lib = B.load()
    assert lib.pa_bank_destroy(None) == B.PA_ERR_NULL
    assert lib.pa_bank_create(B.BANK_ALLOC_FN(), B.BANK_FREE_FN(), None) is None


def test_concurrent_requests_share_one_panel(bank):
    """Host threads asking for the same key at once get one panel."""
    h, fake = bank
    out = []

    def worker():
        for _ in range(50):
            out.append(_get(h, _params(batch=16))[0])

    ts = [threading.Thread(target=worker) for _ in range(8)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert len(set(out)) == 1 and len(fake.allocs) == 1
