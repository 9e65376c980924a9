"""Pins that tie the FP64 oracle to something other than itself.

Each pin takes a loaded oracle library and returns a list of failure messages
(empty = pass), so the same pins run against the real oracle and against
deliberately mutated builds (tests/test_oracle_pins.py checks that every planted
mistake is caught by at least one pin).

What pins what:
  * element decoders  - every E4M3 / E5M2 / FP16 / BF16 code against torch /
                        numpy casts, the E4M3 and E5M2 closed forms, and the OCP
                        format points in tests/golden/e4m3_format_points.txt
                        and tests/golden/e5m2_format_points.txt;
  * whole definition  - brute force on tiny paged inputs against float64
                        torch.nn.functional.scaled_dot_product_attention with an
                        explicit causal mask (an independent library routine);
  * invariants        - uniform scores give the mean of the visible V and
                        lse = log(n); a single visible key returns that key's V;
                        permuting pages together with the block table changes
                        nothing; zero-length rows are exact zeros even when Q is
                        NaN; two keys give sigmoid weights; one-hot V rows expose
                        exactly which keys each verify query sees;
  * row selection     - any list of rows (shuffled, repeated) on any number of
                        threads equals, bit for bit, the same rows of a
                        one-thread evaluation of all rows;
  * prefill entry     - brute force on tiny causal prefills (strided K/V, a
                        context shorter than the query window, q_len ==
                        kv_len) against the same SDPA routine.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import oracle
from helpers import dense_reference, run_oracle, visible
from paged_gqa_decode_split_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "e4m3_format_points.txt")
GOLDEN_E5M2 = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "e5m2_format_points.txt")


def _cmp(name, got, want, atol=0.0, rtol=0.0):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    same = (np.isnan(got) & np.isnan(want)) | (got == want)
    with np.errstate(invalid="ignore"):
        close = np.abs(got - want) <= atol + rtol * np.abs(want)
    bad = ~same & ~close
    if bad.any():
        i = int(np.flatnonzero(bad.ravel())[0])
        return [f"{name}: {int(bad.sum())} mismatches, first at {i}: got {got.ravel()[i]!r} want {want.ravel()[i]!r}"]
    return []


def pin_e4m3_vs_torch(lib):
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return _cmp("e4m3 vs torch float8_e4m3fn", oracle.e4m3_value(codes, lib), want)


def pin_e4m3_closed_form(lib):
    want = []
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            v = math.nan
        elif e == 0:
            v = m * 2.0 ** -9                 # subnormal: m/8 * 2^-6
        else:
            v = (8 + m) * 2.0 ** (e - 10)     # (1 + m/8) * 2^(e-7)
        want.append(-v if s else v)
    return _cmp("e4m3 closed form", oracle.e4m3_value(np.arange(256), lib), want)


def _golden(path, decode, name):
    codes, vals = [], []
    for line in open(path):
        line = line.split("#")[0].strip()
        if line:
            c, v = line.split()
            codes.append(int(c, 16))
            vals.append(float(v))
    got = decode(codes)
    out = _cmp(f"{name} OCP format points", got, vals)
    # the sign of zero is part of the format
    for c, g in zip(codes, got):
        if c in (0x00, 0x80) and math.copysign(1.0, g) != (-1.0 if c == 0x80 else 1.0):
            out.append(f"{name} code {c:#x} has the wrong zero sign")
    return out


def pin_e4m3_golden(lib):
    return _golden(GOLDEN, lambda c: oracle.e4m3_value(c, lib), "e4m3")


def pin_e5m2_vs_torch(lib):
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e5m2).to(torch.float64).numpy()
    return _cmp("e5m2 vs torch float8_e5m2", oracle.e5m2_value(codes, lib), want)


def pin_e5m2_closed_form(lib):
    want = []
    for c in range(256):
        s, e, m = c >> 7, (c >> 2) & 31, c & 3
        if e == 31:
            v = math.inf if m == 0 else math.nan
        elif e == 0:
            v = m * 2.0 ** -16                # subnormal: m/4 * 2^-14
        else:
            v = (4 + m) * 2.0 ** (e - 17)     # (1 + m/4) * 2^(e-15)
        want.append(-v if s else v)
    return _cmp("e5m2 closed form", oracle.e5m2_value(np.arange(256), lib), want)


def pin_e5m2_golden(lib):
    return _golden(GOLDEN_E5M2, lambda c: oracle.e5m2_value(c, lib), "e5m2")


def pin_f16_vs_numpy(lib):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    return _cmp("fp16 vs numpy", oracle.f16_value(bits, lib), bits.view(np.float16).astype(np.float64))


def pin_bf16_vs_torch(lib):
    bits = np.arange(65536, dtype=np.int32).astype(np.uint16)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    return _cmp("bf16 vs torch", oracle.bf16_value(bits, lib), want)


def _tiny(kind, seed, lens, *, Hkv=2, group=3, q_len=4, page_size=16, D=None, layout="separate", base_pad=0):
    spec = wl.small_spec(kind, batch=len(lens), num_kv_heads=Hkv, group=group, q_len=q_len, page_size=page_size,
                         max_ctx_len=max(max(lens), 1), layout=layout, base_pad=base_pad, head_dim=D)
    return wl.generate(spec, seed, ctx_lens=lens)


def _bruteforce(lib, kind, **kw):
    fails = []
    for seed, lens in ((11, [37, 5, 2, 0]), (12, [16, 33, 1])):
        w = _tiny(kind, seed, lens, **kw)
        got, glse = run_oracle(w, lib=lib, num_threads=1)
        ref, rlse = dense_reference(w)
        vis = visible(w)
        fails += _cmp(f"{kind} brute force out (seed {seed})", got[vis], ref[vis], atol=1e-12, rtol=1e-12)
        fails += _cmp(f"{kind} brute force lse (seed {seed})", glse[vis], rlse[vis], atol=1e-12, rtol=1e-12)
        if np.any(got[~vis] != 0.0) or np.any(glse[~vis] != -np.inf):
            fails.append(f"{kind}: rows without keys must be zeros / -inf")
    return fails


def pin_bruteforce_fp8(lib):
    return (_bruteforce(lib, "fp8") +
            _bruteforce(lib, "fp8", Hkv=1, group=6, q_len=8, layout="interleaved", base_pad=8) +
            _bruteforce(lib, "fp8", layout="padded_tokens", base_pad=8))


def pin_bruteforce_e5m2(lib):
    return _bruteforce(lib, "e5m2") + _bruteforce(lib, "e5m2", Hkv=1, group=6, q_len=8, layout="interleaved",
                                                  base_pad=8)


def pin_bruteforce_bf16(lib):
    return _bruteforce(lib, "bf16", Hkv=2, group=4, q_len=1) + _bruteforce(lib, "bf16", D=256)


def pin_bruteforce_f16(lib):
    return _bruteforce(lib, "f16") + _bruteforce(lib, "f16", Hkv=1, group=6, q_len=8, layout="interleaved",
                                                 base_pad=8)


def pin_uniform_mean(lib):
    """Q = 0 makes every score 0: out is the mean of the visible V, lse = log(n)."""
    w = _tiny("fp8", 21, [29, 8, 3], Hkv=2, group=3, q_len=4)
    w.q.zero_()
    got, lse = run_oracle(w, lib=lib, num_threads=1)
    fails = []
    for b, L in enumerate(w.ctx_lens.tolist()):
        for g in range(2):
            from helpers import _elements
            V = _elements(w, "v", b, g, L).numpy()
            for qi in range(4):
                n = L - 4 + qi + 1
                if n <= 0:
                    continue
                for h in range(3 * g, 3 * g + 3):
                    fails += _cmp(f"uniform mean b{b} qi{qi} h{h}", got[b, qi, h], V[:n].mean(0), atol=1e-13)
                    fails += _cmp(f"uniform lse b{b} qi{qi} h{h}", lse[b, qi, h], math.log(n), atol=1e-13)
    return fails


def pin_single_key(lib):
    """With L = q_len, verify query 0 sees exactly key 0 and must return its V."""
    from helpers import _elements
    w = _tiny("fp8", 31, [4, 4], Hkv=2, group=3, q_len=4)
    got, _ = run_oracle(w, lib=lib, num_threads=1)
    fails = []
    for b in range(2):
        for g in range(2):
            v0 = _elements(w, "v", b, g, 1).numpy()[0]
            for h in range(3 * g, 3 * g + 3):
                fails += _cmp(f"single key b{b} h{h}", got[b, 0, h], v0, atol=0.0)
    return fails


def pin_permutation(lib):
    """Moving pages in the pool and rewriting the block table to match leaves
    every output bit unchanged."""
    w = _tiny("fp8", 41, [45, 20], Hkv=2, group=3, q_len=4)
    base, _ = run_oracle(w, lib=lib, num_threads=1)
    s = w.spec
    npg = w.num_pages
    perm = torch.randperm(npg, generator=torch.Generator().manual_seed(5))   # new slot of old page p
    region = npg * s.page_size * s.num_kv_heads * s.head_dim
    kv = w.kv.clone()
    for old in range(npg):
        new = int(perm[old])
        for off in (w.k_offset, w.v_offset):
            src = off + old * w.k_strides[0]
            dst = off + new * w.k_strides[0]
            kv[dst:dst + w.k_strides[0]] = w.kv[src:src + w.k_strides[0]]
    bt = w.block_table.clone()
    m = bt >= 0
    bt[m] = perm[bt[m].long()].to(torch.int32)
    assert region == w.v_offset - w.k_offset
    w2 = wl.Workload(**{**w.__dict__, "kv": kv, "block_table": bt})
    got, _ = run_oracle(w2, lib=lib, num_threads=1)
    if not np.array_equal(got, base):
        return ["page permutation changed the output"]
    return []


def pin_zero_length(lib):
    w = _tiny("fp8", 51, [0, 9, 0], Hkv=2, group=3, q_len=4)
    w.q[0] = float("nan")
    w.q[2] = float("nan")
    got, lse = run_oracle(w, lib=lib, num_threads=1)
    fails = []
    for b in (0, 2):
        if not (np.all(got[b] == 0.0) and np.all(np.signbit(got[b]) == False) and np.all(lse[b] == -np.inf)):
            fails.append(f"zero-length request {b} must give +0.0 and lse -inf")
    if not np.all(np.isfinite(got[1])):
        fails.append("a live request next to NaN-padded slots must stay finite")
    return fails


def pin_two_key(lib):
    """q_len 1, L 2: out = sigmoid(s0 - s1) v0 + sigmoid(s1 - s0) v1."""
    from helpers import _elements
    w = _tiny("fp8", 61, [2, 2], Hkv=1, group=2, q_len=1)
    got, lse = run_oracle(w, lib=lib, num_threads=1)
    fails = []
    D = w.spec.head_dim
    for b in range(2):
        K = _elements(w, "k", b, 0, 2).numpy()
        V = _elements(w, "v", b, 0, 2).numpy()
        for h in range(2):
            q = w.q[b, 0, h].double().numpy()
            s0, s1 = q @ K[0] / math.sqrt(D), q @ K[1] / math.sqrt(D)
            a0 = 1.0 / (1.0 + math.exp(s1 - s0))
            a1 = 1.0 / (1.0 + math.exp(s0 - s1))
            fails += _cmp(f"two-key b{b} h{h}", got[b, 0, h], a0 * V[0] + a1 * V[1], atol=1e-12, rtol=1e-12)
            fails += _cmp(f"two-key lse b{b} h{h}", lse[b, 0, h], max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))),
                          atol=1e-12)
    return fails


def pin_causal_window(lib):
    """BF16 V rows set to one-hot e_j and Q = 0: verify query qi must return
    1/n on exactly coordinates 0..n-1 with n = L - q_len + qi + 1."""
    spec = wl.small_spec("bf16", batch=2, num_kv_heads=1, group=2, q_len=5, page_size=16, max_ctx_len=40,
                         head_dim=64)
    w = wl.generate(spec, 71, ctx_lens=[37, 3])
    w.q.zero_()
    s = spec
    kv = w.kv.clone()
    bt = w.block_table
    for b, L in enumerate(w.ctx_lens.tolist()):
        for j in range(L):
            page = int(bt[b, j // s.page_size])
            start = w.v_offset + page * w.v_strides[0] + (j % s.page_size) * w.v_strides[1]
            row = torch.zeros(s.head_dim, dtype=torch.bfloat16)
            row[j] = 1.0
            kv[start:start + 2 * s.head_dim] = row.view(torch.uint8)
    w = wl.Workload(**{**w.__dict__, "kv": kv})
    got, _ = run_oracle(w, lib=lib, num_threads=1)
    fails = []
    for b, L in enumerate(w.ctx_lens.tolist()):
        for qi in range(s.q_len):
            n = L - s.q_len + qi + 1
            want = np.zeros(s.head_dim)
            if n > 0:
                want[:n] = 1.0 / n
            for h in range(2):
                fails += _cmp(f"causal window b{b} qi{qi} h{h}", got[b, qi, h], want, atol=1e-15)
    return fails


def pin_row_selection_and_threads(lib):
    """Selected rows (shuffled, with repeats) and several threads give, bit
    for bit, the rows of a one-thread evaluation of every row.  Each row is
    one sequential evaluation of the definition, so neither the row order nor
    the thread count may change a bit; this ties the i-th output slot to the
    i-th requested row and keeps each thread's scratch its own."""
    fails = []
    cases = (
        ("tiny", _tiny("fp8", 81, [37, 5, 2, 0], Hkv=2, group=3, q_len=4)),
        ("medium", _tiny("fp8", 82, [1500, 700, 0, 9], Hkv=2, group=3, q_len=8, page_size=32)),
        ("medium bf16", _tiny("bf16", 83, [900, 1200], Hkv=2, group=4, q_len=1, page_size=16)),
    )
    for name, w in cases:
        s = w.spec
        full, full_lse = run_oracle(w, lib=lib, num_threads=1)
        flat = full.reshape(-1, s.head_dim)
        flat_lse = full_lse.reshape(-1)
        n = flat.shape[0]
        rng = np.random.default_rng(7)
        rows = np.concatenate([rng.permutation(n), rng.integers(0, n, n // 2 + 3)]).astype(np.int32)
        rng.shuffle(rows)
        for threads in (2, max(2, oracle.max_threads(lib))):
            got, glse = run_oracle(w, rows=rows, lib=lib, num_threads=threads)
            if got.shape != (rows.size, s.head_dim) or glse.shape != (rows.size,):
                fails.append(f"{name}: row selection returned shapes {got.shape}, {glse.shape}")
                continue
            bad = ~((got == flat[rows]) | (np.isnan(got) & np.isnan(flat[rows]))).all(axis=1)
            bad |= ~((glse == flat_lse[rows]) | (np.isnan(glse) & np.isnan(flat_lse[rows])))
            if bad.any():
                i = int(np.flatnonzero(bad)[0])
                fails.append(f"{name}, {threads} threads: {int(bad.sum())} of {rows.size} selected rows differ "
                             f"from the one-thread rows, first slot {i} (row {int(rows[i])})")
    return fails


def prefill_dense_reference(w: wl.PrefillWorkload):
    """float64 SDPA over the strided K/V views of a prefill workload with an
    explicit causal mask (query i sees keys 0 .. kv_len - q_len + i); rows
    without a key come back as zeros / -inf."""
    s = w.spec
    B, Q, KV, Hq, Hkv, D = s.batch, s.q_len, s.kv_len, s.num_q_heads, s.num_kv_heads, s.head_dim
    G = Hq // Hkv
    q = w.q.detach().cpu().double()
    K, V = w.key_view("k").detach().cpu().double(), w.key_view("v").detach().cpu().double()
    mask = torch.arange(KV)[None, :] <= (KV - Q + torch.arange(Q))[:, None]
    out = np.zeros((B, Q, Hq, D))
    lse = np.full((B, Q, Hq), -np.inf)
    seen = mask.any(dim=1)
    for b in range(B):
        for h in range(Hq):
            kg, vg = K[b, :, h // G], V[b, :, h // G]
            qs = q[b, :, h]
            o = torch.nn.functional.scaled_dot_product_attention(qs[None, None], kg[None, None], vg[None, None],
                                                                 attn_mask=mask[None, None])[0, 0]
            sc = ((qs @ kg.T) / math.sqrt(D)).masked_fill(~mask, float("-inf"))
            ls = torch.logsumexp(sc, dim=-1)
            out[b, seen, h] = o[seen].numpy()
            lse[b, seen, h] = ls[seen].numpy()
    return out, lse


def run_prefill_oracle(w: wl.PrefillWorkload, rows=None, lib=None, num_threads: int = 0):
    s = w.spec

    def bits(t):
        return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)

    return oracle.prefill_attn(q=bits(w.q), k=bits(w.k_buf), v=bits(w.v_buf), k_strides=w.k_strides,
                               v_strides=w.v_strides, kv_len=s.kv_len, num_kv_heads=s.num_kv_heads, rows=rows,
                               num_threads=num_threads, lib=lib)


def pin_prefill_bruteforce(lib):
    """The prefill entry (dense per-request K/V as one page, q_len prefill
    queries) against SDPA on tiny shapes: strided K/V with padded tokens, a
    context shorter than the query window (rows without keys), and q_len ==
    kv_len (plain causal attention)."""
    fails = []
    cases = [(wl.PrefillSpec("pin_a", 2, 37, 300, 6, 2, token_pad=8), 31),
             (wl.PrefillSpec("pin_b", 1, 50, 20, 3, 1), 32),
             (wl.PrefillSpec("pin_c", 1, 64, 64, 4, 2), 33)]
    for spec, seed in cases:
        w = wl.generate_prefill(spec, seed)
        got, glse = run_prefill_oracle(w, lib=lib, num_threads=1)
        ref, rlse = prefill_dense_reference(w)
        fails += _cmp(f"prefill {spec.name} out", got, ref, atol=1e-12, rtol=1e-12)
        fails += _cmp(f"prefill {spec.name} lse", glse, rlse, atol=1e-12, rtol=1e-12)
    return fails


ALL_PINS = [pin_e4m3_vs_torch, pin_e4m3_closed_form, pin_e4m3_golden, pin_e5m2_vs_torch, pin_e5m2_closed_form,
            pin_e5m2_golden, pin_f16_vs_numpy, pin_bf16_vs_torch,
            pin_bruteforce_fp8, pin_bruteforce_e5m2, pin_bruteforce_bf16, pin_bruteforce_f16, pin_uniform_mean, pin_single_key, pin_permutation,
            pin_zero_length, pin_two_key, pin_causal_window, pin_row_selection_and_threads, pin_prefill_bruteforce]
