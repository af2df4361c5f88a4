"""Plant plausible mistakes in copies of the oracle (on the CPU) and check that the pins
catch every one of them: a dropped term, a wrong sign, a wrong index, a swapped operand,
a wrong comparison, a missing rounding rule."""
import os
import types

import numpy as np
import pytest

from oracle_checks import ALL_CHECKS

SRC_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "oracle", "rowpass_oracle.py")

# (name, text in the oracle, replacement)
MUTATIONS = [
    ("temperature_multiplies", "z = x / np.float64(T)", "z = x * np.float64(T)"),
    ("bwd_drops_1_over_T", "g = dlogp * np.asarray(dloss, dtype=np.float64) / np.float64(T)",
     "g = dlogp * np.asarray(dloss, dtype=np.float64)"),
    ("kl_grad_sign", "dkl = beta * (1.0 - np.exp(np.asarray", "dkl = beta * (-1.0 + np.exp(np.asarray"),
    ("kl_value_sign_of_d", "kl = beta * (np.expm1(d) - d)          #", "kl = beta * (np.expm1(d) + d)          #"),
    ("kl_value_dropped", "kl = beta * (np.expm1(d) - d)          #", "kl = beta * np.expm1(d)          #"),
    ("seq_kl_value_sign", "            kl = beta * (np.expm1(d) - d)\n            dkl", "            kl = beta * (np.expm1(d) + d)\n            dkl"),
    ("seq_kl_grad_sign", "dkl = beta * (1.0 - np.exp(d))", "dkl = beta * (np.exp(d) - 1.0)"),
    ("tie_counts_as_clipped", "unclipped_binds = (ratio * A) <= (clipped * A)",
     "unclipped_binds = (ratio * A) < (clipped * A)"),
    ("is_clipped_reversed", "is_clipped = obj_clipped < obj_unclipped", "is_clipped = obj_clipped > obj_unclipped"),
    ("pg_sign", "pg = -np.minimum(obj_unclipped, obj_clipped)", "pg = np.minimum(obj_unclipped, obj_clipped)"),
    ("pg_max_not_min", "pg = -np.minimum(obj_unclipped, obj_clipped)", "pg = -np.maximum(obj_unclipped, obj_clipped)"),
    ("eps_swapped_fwd", "clipped = np.clip(ratio, 1.0 - eps_low, 1.0 + eps_high)\n        obj_unclipped",
     "clipped = np.clip(ratio, 1.0 - eps_high, 1.0 + eps_low)\n        obj_unclipped"),
    ("ratio_inverted", "ratio = np.exp(logp - np.asarray(old_logp, dtype=np.float64))\n        clipped = np.clip(ratio, 1.0 - eps_low, 1.0 + eps_high)\n        unclipped",
     "ratio = np.exp(np.asarray(old_logp, dtype=np.float64) - logp)\n        clipped = np.clip(ratio, 1.0 - eps_low, 1.0 + eps_high)\n        unclipped"),
    ("dpg_missing_ratio", "dpg = np.where(unclipped_binds, -A * ratio, 0.0)", "dpg = np.where(unclipped_binds, -A, 0.0)"),
    ("onehot_wrong_column", "onehot[rows[ok], idx[ok]] = 1.0", "onehot[rows[ok], (idx[ok] + 1) % V] = 1.0"),
    ("grad_sign", "d = g[:, None] * (onehot - p)", "d = g[:, None] * (p - onehot)"),
    ("zero_rows_not_forced", "d[g == 0.0, :] = 0.0", "pass"),
    ("entropy_zero_terms_not_skipped", "np.where(p == 0.0, 0.0, p * (lse[:, None] - z))", "p * (lse[:, None] - z)"),
    ("entropy_sign", "np.where(p == 0.0, 0.0, p * (lse[:, None] - z))", "np.where(p == 0.0, 0.0, p * (z - lse[:, None]))"),
    ("lse_drops_max", "lse = (m + np.log(s))[..., 0]", "lse = np.log(s)[..., 0]"),
    ("linear_grad_h_scaled", "grad_h = dx @ W\n", "grad_h = dx @ W / T\n"),
    ("linear_grad_W_sign", "grad_W = dx.T @ h\n", "grad_W = -(dx.T @ h)\n"),
    ("linear_head_scaled", "x = h @ W.T\n", "x = h @ W.T * 1.01\n"),
    ("all_neginf_row_not_handled", "m = np.where(np.isneginf(m), 0.0, m)", "pass"),
    ("lse_no_shift", "s = np.sum(np.exp(z - m), axis=-1, keepdims=True)\n        lse = (m + np.log(s))[..., 0]",
     "s = np.sum(np.exp(z), axis=-1, keepdims=True)\n        lse = np.log(s)[..., 0]"),
    ("logp_sign_of_lse", "logp = z[rows, np.asarray(idx, dtype=np.int64)] - lse",
     "logp = z[rows, np.asarray(idx, dtype=np.int64)] + lse"),
    ("mask_ignored_in_loss", '"loss": np.where(mask, loss, z),', '"loss": loss,'),
    ("entropy_bwd_sign_of_H", "d = g[:, None] * np.where(p == 0.0, 0.0, p * (logp + H[:, None]))",
     "d = g[:, None] * np.where(p == 0.0, 0.0, p * (logp - H[:, None]))"),
    ("entropy_bwd_drops_T", "g = -np.asarray(dentropy, dtype=np.float64) / np.float64(T)",
     "g = -np.asarray(dentropy, dtype=np.float64)"),
    ("entropy_zero_rows_not_forced", "    d[g == 0.0] = 0.0 ", "    pass  "),
    ("seq_ratio_not_length_normalised", "np.where(m, logp - old, 0.0).sum(axis=1) / np.maximum(n, 1)",
     "np.where(m, logp - old, 0.0).sum(axis=1)"),
    ("seq_dpg_missing_weight", "dlogp = (W * dpg)[:, None] + dkl * dl", "dlogp = dpg[:, None] + dkl * dl"),
    ("seq_kl_grad_unweighted", "dlogp = (W * dpg)[:, None] + dkl * dl", "dlogp = (W * dpg)[:, None] + dkl"),
    ("bf16_truncates", "q = np.rint(np.ldexp(a, -unit_exp))", "q = np.floor(np.ldexp(a, -unit_exp))"),
    ("bf16_ties_away", "q = np.rint(np.ldexp(a, -unit_exp))", "q = np.floor(np.ldexp(a, -unit_exp) + 0.5)"),
    ("bf16_mantissa_bits", "_BF16_MANT_BITS = 7 ", "_BF16_MANT_BITS = 8 "),
    ("bf16_no_subnormals", "unit_exp = np.maximum(e - 1 - _BF16_MANT_BITS, _BF16_MIN_EXP - _BF16_MANT_BITS)",
     "unit_exp = e - 1 - _BF16_MANT_BITS"),
    ("bf16_decode_shift", "astype(np.uint32) << np.uint32(16)", "astype(np.uint32) << np.uint32(15)"),
]


def _mutant(old, new):
    src = open(SRC_PATH).read()
    assert src.count(old) == 1, f"mutation anchor not unique/found: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(name, old, new):
    mod = _mutant(old, new)
    caught = []
    with np.errstate(all="ignore"):
        for check in ALL_CHECKS:
            try:
                check(mod)
            except Exception as e:  # an assertion or a crash both count as caught
                caught.append(check.__name__)
    assert caught, f"no pin catches mutation {name}"
