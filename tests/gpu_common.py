"""Shared helpers of the GPU tests: tolerance checks against the FP64 oracle."""
from __future__ import annotations

import numpy as np
import torch

from helpers import run_oracle, visible

# Tolerances against the FP64 oracle.  FP16 outputs: max-abs 2e-3 and rel-L2
# 3e-3 over every row that sees a key.  BF16 outputs keep 8 significant bits,
# so rounding alone moves a value by up to 2^-8 of its magnitude (3.9e-3 for
# |x| in [1, 2)); their element bound adds that rounding term to 2e-3.
MAX_ABS = 2e-3
REL_L2 = 3e-3
BF16_REL_ROUND = 2.0 ** -8


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_full(w, out: torch.Tensor, lse: torch.Tensor | None = None, oracle_threads: int = 0):
    """Every row against the oracle: visible rows within tolerance, rows with
    no key exactly +0.0.  Returns (max_abs, rel_l2)."""
    ref, rlse = run_oracle(w.to("cpu"), num_threads=oracle_threads)
    got = to_f64(out)
    vis = visible(w.to("cpu"))
    return _compare(got, ref, vis, lse, rlse, bf16=out.dtype == torch.bfloat16)


def check_rows(w, out: torch.Tensor, rows: np.ndarray, oracle_threads: int = 0):
    """Sampled flat rows ((b*q_len + qi)*Hq + h) against the oracle."""
    s = w.spec
    ref, _ = run_oracle(w.to("cpu"), rows=rows, num_threads=oracle_threads)
    got = to_f64(out).reshape(-1, s.head_dim)[rows]
    vis = visible(w.to("cpu")).reshape(-1)[rows]
    return _compare(got, ref, vis, None, None, bf16=out.dtype == torch.bfloat16)


def _compare(got, ref, vis, lse, rlse, bf16=False, rel_elem=0.0):
    """rel_elem adds rel_elem * |ref| to the FP16 element bound (outputs whose
    magnitude is set by one dominant key: FP16 output rounding and the FP16
    rounding of that key's weight each move it by up to 2^-11 of |ref|)."""
    assert np.all(np.isfinite(got)), "non-finite output"
    zero_rows = got[~vis]
    assert np.all(zero_rows == 0.0) and not np.any(np.signbit(zero_rows)), "rows without keys must be +0.0"
    if not vis.any():
        return 0.0, 0.0
    d = got[vis] - ref[vis]
    max_abs = float(np.abs(d).max())
    rel_l2 = float(np.linalg.norm(d) / max(np.linalg.norm(ref[vis]), 1e-30))
    if bf16:
        excess = np.abs(d) - (MAX_ABS + BF16_REL_ROUND * np.abs(ref[vis]))
        assert excess.max() <= 0, f"BF16 element error {max_abs:.3e} beyond 2e-3 + 2^-8 |ref|"
    elif rel_elem > 0.0:
        excess = np.abs(d) - (MAX_ABS + rel_elem * np.abs(ref[vis]))
        assert excess.max() <= 0, f"FP16 element error {max_abs:.3e} beyond 2e-3 + {rel_elem:.3g} |ref|"
    else:
        assert max_abs <= MAX_ABS, f"max abs error {max_abs:.3e} > {MAX_ABS}"
    assert rel_l2 <= REL_L2, f"relative L2 error {rel_l2:.3e} > {REL_L2}"
    if lse is not None:
        gl = to_f64(lse)
        assert np.all(gl[~vis] == -np.inf)
        lerr = float(np.abs(gl[vis] - rlse[vis]).max())
        assert lerr <= 1e-3, f"lse error {lerr:.3e}"
    return max_abs, rel_l2
