"""Pins of the comparison rule (oracle/compare.py) that every float parity
claim goes through.

The rule is the tolerance the problem statement fixes for this path: out
within relative L2 1e-2 and max |diff| 2e-2 of the oracle rounded to bf16,
lse within 2e-3 on finite entries, -inf exactly where the oracle row is
empty (with all-zero out bits there), no NaN anywhere.  Each check below
feeds the comparator a result with exactly one rule broken -- just past its
threshold -- and requires a rejection, and the same result just inside the
threshold, which must pass.  The mutation test at the end plants plausible
mistakes in the comparator's own source (an inverted comparison, a dropped
check, a wrong mask, a wrong norm) and requires these checks to catch each.
CPU only."""
import inspect
import math

import numpy as np
import pytest
import torch

import oracle.compare as compare_mod
from oracle.compare import LSE_ABS, OUT_MAX_ABS, OUT_REL_L2, bf16_round, compare_out_lse


def _case(seed=0, T=3, H=4, empty=((1, 2),)):
    """A plausible oracle result: out ~ N(0, 1) [T, H, 512] float64, lse
    finite, with the listed (token, head) rows empty (out 0, lse -inf)."""
    rng = np.random.default_rng(seed)
    out = rng.standard_normal((T, H, 512))
    lse = rng.uniform(-3.0, 8.0, size=(T, H))
    for t, h in empty:
        out[t, h] = 0.0
        lse[t, h] = -np.inf
    return out, lse


def _gpu_like(out_ref, lse_ref):
    """What a perfect kernel returns: out rounded to bf16 (as a torch bf16
    tensor) and lse as fp32."""
    o = torch.from_numpy(out_ref).to(torch.bfloat16)
    l = torch.from_numpy(lse_ref).to(torch.float32)
    return o, l


def _rejects(cmp, *args):
    try:
        cmp(*args)
    except AssertionError:
        return True
    return False


# Each check returns True when the comparator behaves as the rule says.
def check_exact_result_passes(cmp):
    out, lse = _case()
    o, l = _gpu_like(out, lse)
    return not _rejects(cmp, o, l, out, lse)


def check_one_element_off_by_max_abs(cmp):
    out, lse = _case(1)
    ref = bf16_round(out)
    bad = ref.copy()
    bad[0, 0, 7] += 1.05 * OUT_MAX_ABS
    ok = ref.copy()
    ok[0, 0, 7] += 0.95 * OUT_MAX_ABS
    return _rejects(cmp, bad, lse, out, lse) and not _rejects(cmp, ok, lse, out, lse)


def check_diffuse_noise_by_rel_l2(cmp):
    """Noise of fixed magnitude delta on every element: relative L2 just
    above (then below) 1e-2 while max |diff| stays well under 2e-2."""
    out, lse = _case(2, empty=())
    ref = bf16_round(out)
    rng = np.random.default_rng(22)
    sign = np.where(rng.random(out.shape) < 0.5, -1.0, 1.0)
    norm = np.linalg.norm(ref)
    delta_bad = 1.1 * OUT_REL_L2 * norm / math.sqrt(out.size)
    delta_ok = 0.9 * OUT_REL_L2 * norm / math.sqrt(out.size)
    assert delta_bad < 0.6 * OUT_MAX_ABS
    return (_rejects(cmp, ref + sign * delta_bad, lse, out, lse)
            and not _rejects(cmp, ref + sign * delta_ok, lse, out, lse))


def check_one_lse_off(cmp):
    out, lse = _case(3)
    o, l = _gpu_like(out, lse)
    l64 = lse.astype(np.float32).astype(np.float64)
    bad = l64.copy()
    bad[2, 1] = lse[2, 1] + 1.05 * LSE_ABS
    ok = l64.copy()
    ok[2, 1] = lse[2, 1] - 0.95 * LSE_ABS
    return _rejects(cmp, o, bad, out, lse) and not _rejects(cmp, o, ok, out, lse)


def check_nan_in_out(cmp):
    out, lse = _case(4)
    o, l = _gpu_like(out, lse)
    o[2, 3, 100] = float("nan")
    return _rejects(cmp, o, l, out, lse)


def check_nan_in_lse(cmp):
    out, lse = _case(5)
    o, l = _gpu_like(out, lse)
    l[0, 0] = float("nan")
    return _rejects(cmp, o, l, out, lse)


def check_neg_inf_only_on_gpu(cmp):
    out, lse = _case(6)
    o, l = _gpu_like(out, lse)
    l[0, 3] = -math.inf
    o[0, 3] = 0
    return _rejects(cmp, o, l, out, lse)


def check_neg_inf_only_in_oracle(cmp):
    out, lse = _case(7)
    o, l = _gpu_like(out, lse)
    l[1, 2] = 0.5  # the oracle row (1, 2) is empty
    return _rejects(cmp, o, l, out, lse)


def check_neg_inf_on_gpu_where_oracle_out_is_zero(cmp):
    """The oracle row is not empty (finite lse) but its out is exactly zero
    (all its value rows are zero); a result that reports it as the empty
    identity (0, -inf) has the right out and must still be rejected."""
    out, lse = _case(12)
    out[2, 0] = 0.0
    o, l = _gpu_like(out, lse)
    l[2, 0] = -math.inf
    return _rejects(cmp, o, l, out, lse)


def check_empty_row_with_one_nonzero(cmp):
    """One non-zero element in an empty row, inside every float tolerance:
    rejected both as a bf16 tensor and as a plain float64 array (the second
    form has no bit pattern to inspect, only values)."""
    out, lse = _case(8)
    o, l = _gpu_like(out, lse)
    o[1, 2, 300] = 1e-3
    o64 = bf16_round(out)
    o64[1, 2, 300] = 1e-3
    return _rejects(cmp, o, l, out, lse) and _rejects(cmp, o64, l, out, lse)


def check_empty_row_with_negative_zero_bits(cmp):
    out, lse = _case(9)
    o, l = _gpu_like(out, lse)
    o[1, 2, 5] = -0.0
    assert o.view(torch.int16)[1, 2, 5].item() != 0
    return _rejects(cmp, o, l, out, lse)


def check_shape_mismatch(cmp):
    out, lse = _case(10)
    o, l = _gpu_like(out, lse)
    return (_rejects(cmp, o[:, :3], l[:, :3], out, lse)
            and _rejects(cmp, o[..., :256], l, out, lse)
            and _rejects(cmp, o, l[:, :3], out, lse)
            and _rejects(cmp, o, l, out[:2], lse[:2]))


def check_empty_rows_exact_pass(cmp):
    """Many empty rows, all exact: must pass (the rule must not reject the
    identity itself)."""
    out, lse = _case(11, T=4, H=3, empty=((0, 0), (0, 1), (3, 2), (2, 0)))
    o, l = _gpu_like(out, lse)
    return not _rejects(cmp, o, l, out, lse)


CHECKS = [
    check_exact_result_passes,
    check_one_element_off_by_max_abs,
    check_diffuse_noise_by_rel_l2,
    check_one_lse_off,
    check_nan_in_out,
    check_nan_in_lse,
    check_neg_inf_only_on_gpu,
    check_neg_inf_only_in_oracle,
    check_neg_inf_on_gpu_where_oracle_out_is_zero,
    check_empty_row_with_one_nonzero,
    check_empty_row_with_negative_zero_bits,
    check_shape_mismatch,
    check_empty_rows_exact_pass,
]


@pytest.mark.parametrize("check", CHECKS, ids=lambda f: f.__name__)
def test_comparator_rule(check):
    assert check(compare_out_lse)


def test_tolerance_constants_are_the_stated_ones():
    assert (OUT_REL_L2, OUT_MAX_ABS, LSE_ABS) == (1e-2, 2e-2, 2e-3)


# ----------------------------------------------------------------- mutants
# Plausible mistakes in the comparator's source, each a (pattern, replacement)
# applied once to oracle/compare.py's text.  Dropping one of the two explicit
# NaN checks is not among them: a NaN in out or lse also fails the error
# bounds (NaN compares false) or the -inf / empty-row checks, so such a
# mutant accepts nothing the comparator rejects.  Nor is dropping the lse
# shape check: the -inf pattern comparison (np.array_equal) already rejects
# arrays of different shapes.
MUTANTS = {
    "lse_comparison_inverted": ("assert lse_err <= LSE_ABS", "assert lse_err >= 0 or lse_err <= LSE_ABS"),
    "rel_l2_check_dropped": ("assert rel_l2 <= OUT_REL_L2", "assert rel_l2 == rel_l2"),
    "max_abs_check_dropped": ("assert max_abs <= OUT_MAX_ABS", "assert max_abs == max_abs"),
    "max_abs_uses_mean": ("max_abs = float(np.abs(diff).max())", "max_abs = float(np.abs(diff).mean())"),
    "rel_l2_against_gpu_norm": ("denom = float(np.linalg.norm(o_ref))", "denom = float(np.linalg.norm(o)) * 10"),
    "empty_mask_from_gpu": ("empty = np.isneginf(l_ref)", "empty = np.isneginf(l)"),
    "neg_inf_pattern_dropped": ("assert np.array_equal(np.isneginf(l), empty)", "assert True"),
    "empty_bits_dropped": ("assert np.all(bits == 0)", "assert True"),
    "empty_zero_check_dropped": ("assert np.all(o[empty] == 0.0)", "assert True"),
    "lse_only_first_row": ("lse_err = float(np.abs(l[fin] - l_ref[fin]).max())",
                           "lse_err = float(np.abs(l[:1][fin[:1]] - l_ref[:1][fin[:1]]).max(initial=0))"),
    "no_bf16_round_of_ref": ("o_ref = bf16_round(out_ref)", "o_ref = np.asarray(out_ref, dtype=np.float64) * 1.02"),
    "out_shape_check_dropped": ('assert o.shape == o_ref.shape, f"{where}: out shape {o.shape} vs {o_ref.shape}"',
                                "pass"),
    "lse_tolerance_typo": ("LSE_ABS = 2e-3", "LSE_ABS = 2e-2"),
    "max_abs_tolerance_typo": ("OUT_MAX_ABS = 2e-2", "OUT_MAX_ABS = 2e-1"),
}


def _mutant(name):
    src = inspect.getsource(compare_mod)
    pat, rep = MUTANTS[name]
    assert src.count(pat) == 1, f"mutant {name}: pattern not found exactly once"
    ns = {}
    exec(compile(src.replace(pat, rep), f"<mutant {name}>", "exec"), ns)
    return ns["compare_out_lse"]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_rule_checks_catch_planted_comparator_mistake(name):
    cmp = _mutant(name)
    failed = []
    for check in CHECKS:
        try:
            good = check(cmp)
        except Exception:  # a mutant that crashes is caught too
            good = False
        if not good:
            failed.append(check.__name__)
    assert failed, f"no rule check catches mutant {name}"
