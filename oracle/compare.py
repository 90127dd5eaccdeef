"""Comparison rules between the CUDA path and the oracle (test infrastructure).

Tolerances are the ones the problem statement fixes for this path:
  - indices and valid counts: bit-exact
  - empty rows: out all zero bits and lse == -inf exactly
  - out: the oracle rounded to bf16 (round-to-nearest-even); relative L2 over
    the compared tensor <= 1e-2 and max |diff| <= 2e-2
  - lse: |diff| <= 2e-3 on finite entries; -inf matches -inf; no NaN anywhere
"""
from __future__ import annotations

import numpy as np
import torch

OUT_REL_L2 = 1e-2
OUT_MAX_ABS = 2e-2
LSE_ABS = 2e-3


def bf16_round(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, dtype=np.float64)).to(torch.bfloat16).to(
        torch.float64).numpy()


def to_f64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu").to(torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def compare_out_lse(out_gpu, lse_gpu, out_ref, lse_ref, where: str = ""):
    """Raise AssertionError with a readable message when a rule is broken.
    Returns a dict of the measured errors."""
    o = to_f64(out_gpu)
    l = to_f64(lse_gpu)
    o_ref = bf16_round(out_ref)
    l_ref = np.asarray(lse_ref, dtype=np.float64)
    assert o.shape == o_ref.shape, f"{where}: out shape {o.shape} vs {o_ref.shape}"
    assert l.shape == l_ref.shape, f"{where}: lse shape {l.shape} vs {l_ref.shape}"
    assert not np.isnan(o).any(), f"{where}: NaN in out"
    assert not np.isnan(l).any(), f"{where}: NaN in lse"
    empty = np.isneginf(l_ref)
    assert np.array_equal(np.isneginf(l), empty), f"{where}: -inf pattern differs"
    if empty.any():
        assert np.all(o[empty] == 0.0), f"{where}: empty rows not zero"
        if isinstance(out_gpu, torch.Tensor):
            bits = out_gpu.detach().cpu().view(torch.int16).numpy()[empty]
            assert np.all(bits == 0), f"{where}: empty rows not all-zero bits"
    fin = ~empty
    lse_err = float(np.abs(l[fin] - l_ref[fin]).max()) if fin.any() else 0.0
    diff = o - o_ref
    denom = float(np.linalg.norm(o_ref))
    rel_l2 = float(np.linalg.norm(diff) / denom) if denom > 0 else float(np.linalg.norm(diff))
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    assert lse_err <= LSE_ABS, f"{where}: lse max abs err {lse_err:.3e} > {LSE_ABS}"
    assert rel_l2 <= OUT_REL_L2, f"{where}: out rel L2 {rel_l2:.3e} > {OUT_REL_L2}"
    assert max_abs <= OUT_MAX_ABS, f"{where}: out max abs err {max_abs:.3e} > {OUT_MAX_ABS}"
    return {"lse_max_abs": lse_err, "out_rel_l2": rel_l2, "out_max_abs": max_abs}
