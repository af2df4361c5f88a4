"""Helpers for comparing the CUDA path with the oracle.

Tolerances (written out here, used by every parity test):

* logp, lse, entropy, loss, kl:  |gpu - oracle| <= 1e-5 + 1e-5 * |oracle|; NaN where the
  oracle is NaN; masked-row outputs are +0.0 bit for bit.
* bf16 dlogits: within 1 bf16 ulp of the oracle value rounded to nearest even directly
  from fp64; where |oracle| < 2^-126 (below the smallest normal) the GPU value may be any
  bf16 below 2^-126 in magnitude, zero included (the exponential flushes there).
* fp32 dlogits: |gpu - oracle| <= (1e-5 + rho) * |oracle| + 1e-7 * |g|, with g the row
  factor and rho the row's propagated input error (below).
* rows whose row factor g is exactly 0 in the oracle: every element +0.0 bit for bit.
* is_clipped: equal.

The backward takes logp and lse from the GPU forward (fp32).  Every element of a row is
g * (1[j == idx] - p_j), so an error in lse scales the row by e^{dlse} and an error in
logp moves g by dg/dlogp * dlogp, with |dg/dlogp| <= (|A| ratio + beta e^{d}) |dloss| / T.
The row's relative error budget is therefore

    rho = |dlse| + (S |dlogp| + 3e-7 (|A| ratio + |kl'|) |dloss| / T) / |g| + 1e-6,

with dlse, dlogp the forward's actual deviations from the oracle on that row.  Where
rho > 2^-10 (a quarter of a bf16 ulp) fp32 cannot pin the row to 1 bf16 ulp: such rows are
"ambiguous" (e.g. KL-only rows with a tiny ref - logp, or policy and KL terms that
cancel), as are rows whose ratio lies within 1e-5 (relative) of a clip boundary on a
token with A != 0 (fp32 and fp64 may take different branches).  Ambiguous rows are
excluded from the element checks, their count is asserted small, and they still pass the
row-sum invariant.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle

SCALAR_RTOL = 1e-5
SCALAR_ATOL = 1e-5
TINY = 2.0 ** -126


def rows_f64(t: torch.Tensor) -> np.ndarray:
    """[k, V] bf16/fp32 tensor (any device) -> float64 numpy, exactly."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return oracle.bf16_bits_to_fp64(t.view(torch.int16).numpy().view(np.uint16))
    return oracle.decode_logits(t.numpy(), "fp32")


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_scalar_close(gpu, orc, what, rtol=SCALAR_RTOL, atol=SCALAR_ATOL, where=None):
    g = np.asarray(gpu.detach().cpu().numpy() if isinstance(gpu, torch.Tensor) else gpu, dtype=np.float64)
    o = np.asarray(orc, dtype=np.float64)
    if where is not None:
        g, o = g[where], o[where]
    nan_o = np.isnan(o)
    assert np.array_equal(np.isnan(g), nan_o), f"{what}: NaN pattern differs"
    inf_o = np.isinf(o)
    assert np.array_equal(g[inf_o], o[inf_o]), f"{what}: inf values differ"
    fin = ~nan_o & ~inf_o
    err = np.abs(g[fin] - o[fin])
    tol = atol + rtol * np.abs(o[fin])
    bad = err > tol
    assert not np.any(bad), (f"{what}: {int(bad.sum())} of {fin.sum()} outside tolerance; worst "
                             f"|diff| {err.max():.3g} at oracle {o[fin][np.argmax(err - tol)]:.6g}")


def assert_plus_zero(t: torch.Tensor, what: str):
    """Every element is +0.0 (bit pattern 0)."""
    t = t.detach()
    if t.dtype == torch.bfloat16:
        nz = int((t.contiguous().view(torch.int16) != 0).sum())
    elif t.dtype == torch.float32:
        nz = int((t.contiguous().view(torch.int32) != 0).sum())
    else:
        nz = int((t != 0).sum())
    assert nz == 0, f"{what}: {nz} elements are not +0.0"


def _bf16_key(b: np.ndarray) -> np.ndarray:
    b = b.astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def assert_bf16_grad_close(gpu_bits: np.ndarray, orc: np.ndarray, what: str):
    orc_bits = oracle.round_to_bf16_bits(orc)
    nan_o = np.isnan(orc)
    nan_g = ((gpu_bits & 0x7F80) == 0x7F80) & ((gpu_bits & 0x007F) != 0)
    assert np.array_equal(nan_o, nan_g), f"{what}: NaN pattern differs"
    d = np.abs(_bf16_key(gpu_bits) - _bf16_key(orc_bits))
    tiny_ok = (np.abs(orc) < TINY) & ((gpu_bits & 0x7F80) == 0)
    ok = (d <= 1) | tiny_ok | nan_o
    if not np.all(ok):
        k = np.argwhere(~ok)[0]
        raise AssertionError(f"{what}: {int((~ok).sum())} elements beyond 1 bf16 ulp; first at {tuple(k)}: "
                             f"gpu {gpu_bits[tuple(k)]:#06x} oracle {orc_bits[tuple(k)]:#06x} ({orc[tuple(k)]:.8g})")


def assert_fp32_grad_close(gpu: np.ndarray, orc: np.ndarray, g: np.ndarray, rho: np.ndarray, what: str):
    gpu = np.asarray(gpu, dtype=np.float64)
    nan_o = np.isnan(orc)
    assert np.array_equal(nan_o, np.isnan(gpu)), f"{what}: NaN pattern differs"
    tol = (1e-5 + rho[:, None]) * np.abs(orc) + 1e-7 * np.abs(g)[:, None]
    tiny_ok = (np.abs(orc) < TINY) & (np.abs(gpu) < TINY)
    err = np.abs(gpu - orc)
    bad = (err > tol) & ~nan_o & ~tiny_ok
    assert not np.any(bad), f"{what}: {int(bad.sum())} elements outside tolerance, worst {err[bad].max():.3g}"


def assert_grad_rows(gpu_rows: torch.Tensor, orc_rows: np.ndarray, g: np.ndarray, skip: np.ndarray, what: str,
                     rho=None):
    """gpu_rows [k, V] vs oracle fp64 [k, V]; rows with g == 0 must be +0.0 exactly;
    rows flagged in `skip` are only checked for the row-sum invariant."""
    rho = np.full(len(g), 1e-6) if rho is None else np.asarray(rho, dtype=np.float64)
    zero = (g == 0.0) & ~skip
    if np.any(zero):
        assert_plus_zero(gpu_rows[torch.from_numpy(np.nonzero(zero)[0]).to(gpu_rows.device)], f"{what} zero rows")
    live = ~zero & ~skip
    if np.any(live):
        sel = np.nonzero(live)[0]
        sub = gpu_rows[torch.from_numpy(sel).to(gpu_rows.device)]
        if gpu_rows.dtype == torch.bfloat16:
            assert_bf16_grad_close(bf16_bits(sub), orc_rows[sel], what)
        else:
            assert_fp32_grad_close(sub.cpu().numpy(), orc_rows[sel], g[sel], rho[sel], what)
    if np.any(skip):
        sel = np.nonzero(skip)[0]
        sub = rows_f64(gpu_rows[torch.from_numpy(sel).to(gpu_rows.device)])
        V = sub.shape[1]
        bound = np.abs(g[sel]) * (1e-4 + V * 2.0 ** -8 if gpu_rows.dtype == torch.bfloat16 else 1e-4) + 1e-30
        assert np.all(np.abs(sub.sum(axis=1)) <= bound), f"{what}: ambiguous rows break the row-sum invariant"


def row_error_budget(g, ratio, adv_row, beta, logp_orc, ref, dloss, T, dlogp, dlse):
    """rho of the module docstring, per row (numpy)."""
    g = np.abs(np.asarray(g, dtype=np.float64))
    A = np.abs(np.asarray(adv_row, dtype=np.float64))
    ratio = np.nan_to_num(np.asarray(ratio, dtype=np.float64), nan=0.0, posinf=1e300)
    scale = np.abs(np.asarray(dloss, dtype=np.float64)) / T
    if beta != 0.0 and ref is not None:
        d = np.asarray(ref, dtype=np.float64) - np.asarray(logp_orc, dtype=np.float64)
        kl_sens = beta * np.exp(d)
        kl_grad = beta * np.abs(np.expm1(d))
    else:
        kl_sens = kl_grad = np.zeros_like(g)
    S = (A * ratio + kl_sens) * scale
    num = S * np.abs(dlogp) + 3e-7 * (A * ratio + kl_grad) * scale
    with np.errstate(divide="ignore", invalid="ignore"):
        rho = np.abs(dlse) + np.where(g > 0, num / np.where(g > 0, g, 1.0), 0.0) + 1e-6
    return rho


def ambiguous_rows(ratio, adv_row, mask, eps_low, eps_high, rho=None):
    """Rows where an fp32 evaluation may legitimately take another branch than fp64, or
    where the propagated input error exceeds a quarter bf16 ulp."""
    ratio = np.asarray(ratio, dtype=np.float64)
    A = np.asarray(adv_row, dtype=np.float64)
    live = np.ones(ratio.shape, bool) if mask is None else (np.asarray(mask) != 0)
    lo, hi = 1.0 - eps_low, 1.0 + eps_high
    amb = live & (A != 0) & ((np.abs(ratio - lo) <= 1e-5 * lo) | (np.abs(ratio - hi) <= 1e-5 * hi))
    if rho is not None:
        amb |= live & (np.asarray(rho) > 2.0 ** -10)
    return amb


def f32(v) -> float:
    """A Python float holding exactly the fp32 value the kernels receive."""
    return float(np.float32(v))
