"""Helpers shared by the GPU parity tests: tensor <-> oracle bit arrays and
the comparison rule.  No attention or paging arithmetic lives here."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# max |gpu - oracle| allowed on the attention output, by output / cache type
TOL = {"f16": 2e-3, "bf16": 8e-3, "e4m3": 3e-2}

ACT_CODE = {torch.float16: oracle.F16, torch.bfloat16: oracle.BF16}


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


def assert_attention_close(got: torch.Tensor, want: np.ndarray, tol: float, rounding_slack: bool = False):
    """max |got - want| <= tol (plus half an output ulp when asked: for tiny
    contexts whose outputs reach magnitudes where rounding to 16 bits alone
    exceeds the tolerance)."""
    g = got.detach().float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g)), "non-finite output"
    err = np.abs(g - want)
    bound = tol + (half_ulp(want, got.dtype) if rounding_slack else 0.0)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), f"max err {err.max():.3e} (at {worst}: got {g[worst]}, want {want[worst]}), tol {tol}"
    return float(err.max())


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
