"""Helpers shared by the GPU parity tests: tensor <-> oracle bit arrays and
the comparison rule.  No attention or paging arithmetic lives here.

The comparison rule (attention outputs against the float64 oracle):

    |got - want| <= tol                    for every element, where tol is
                                           2e-3 (binary16 output), 8e-3
                                           (bfloat16 output) or 3e-2 (E4M3
                                           cache, dequantised values)

with one exception.  The kernel must round its result to the 16-bit output
type, and for large outputs that single rounding is by itself comparable to
the tolerance: half an output ulp is 2^-8 |x| for bfloat16 (7.8e-3 already
at |x| = 2) and 2^-11 |x| for binary16.  An element whose half-ulp exceeds
tol / 2 is therefore allowed tol + half an ulp of the oracle's value; every
other element is held to the plain tol.  Only short contexts (a few tokens,
where the output is close to a single value row) produce such magnitudes.
Every call records its largest error as a fraction of the plain tol and how
many elements needed the extra half-ulp; the session prints the table.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle

# max |gpu - oracle| allowed on the attention output, by output / cache type
TOL = {"f16": 2e-3, "bf16": 8e-3, "e4m3": 3e-2}

ACT_CODE = {torch.float16: oracle.F16, torch.bfloat16: oracle.BF16}

# (test id, max |err|, tol, max |err| / tol over the elements held to the plain tol,
#  max |err| / bound over all elements, elements, elements given the half-ulp)
RESULTS: list[tuple[str, float, float, float, float, int, int]] = []


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw element bits of a tensor as a numpy array (uint16 or uint8)."""
    t = t.detach().contiguous().cpu()
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return t.view(torch.uint8).numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def half_ulp(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """Half a unit in the last place of the output type at |x| (the final rounding)."""
    mant = 10 if dtype == torch.float16 else 7
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -14)))
    return 0.5 * 2.0 ** (e - mant)


def rounding_allowance(want: np.ndarray, dtype: torch.dtype, tol: float) -> np.ndarray:
    """Per-element extra allowance: half an output ulp where that half-ulp is
    more than tol / 2, else 0."""
    h = half_ulp(want, dtype)
    return np.where(h > tol / 2, h, 0.0)


def assert_attention_close(got: torch.Tensor, want: np.ndarray, tol: float, label: str = ""):
    """Every element within tol of the oracle (plus half an output ulp only on
    elements whose own rounding to the output type is more than tol / 2)."""
    g = got.detach().float().cpu().numpy().astype(np.float64)
    assert g.shape == want.shape, f"shape {g.shape} vs oracle {want.shape}"
    assert np.all(np.isfinite(g)), "non-finite output"
    err = np.abs(g - want)
    extra = rounding_allowance(want, got.dtype, tol)
    bound = tol + extra
    n_extra = int(np.count_nonzero(extra))
    worst_abs = float(err.max()) if err.size else 0.0
    plain = err[extra == 0]
    frac_plain = float(plain.max()) / tol if plain.size else 0.0
    frac_bound = float((err / bound).max()) if err.size else 0.0
    test_id = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    if label and label not in test_id:
        test_id += f"[{label}]"
    RESULTS.append((test_id, worst_abs, tol, frac_plain, frac_bound, err.size, n_extra))
    if err.size:
        worst = np.unravel_index(np.argmax(err - bound), err.shape)
        assert np.all(err <= bound), (f"max err {worst_abs:.3e} (worst vs its bound at {worst}: got {g[worst]}, "
                                      f"want {want[worst]}, bound {bound[worst]:.3e}), tol {tol}")
    return worst_abs


def compact_pool(k_cache: torch.Tensor, v_cache: torch.Tensor, tables: np.ndarray, lens: np.ndarray, bs: int):
    """Copy only the blocks the given sequences use to the host; return the
    compacted pools and the tables renumbered into them."""
    used = sorted({int(b) for row, L in zip(tables, lens) for b in row[: -(-int(L) // bs)]})
    remap = {b: i for i, b in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.long, device=k_cache.device)
    kc = k_cache.index_select(0, idx).cpu()
    vc = v_cache.index_select(0, idx).cpu()
    t2 = np.zeros_like(tables)
    for i, (row, L) in enumerate(zip(tables, lens)):
        for j in range(-(-int(L) // bs)):
            t2[i, j] = remap[int(row[j])]
    return kc, vc, t2
