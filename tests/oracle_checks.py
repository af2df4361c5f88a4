"""Pins for the fp64 oracle: checks against facts that do not come from the oracle.

Every check takes the oracle module as ``orc`` and raises AssertionError when the
oracle disagrees with something the pages or the mathematics fix:

* brute force at high precision (mpmath with 50 digits, or long double) on tiny rows,
  with no max-shift;
* closed forms (V = 2, all-equal rows, two-level rows, the textbook cases of the
  PPO clipped objective, the k3 KL estimator at d = +-ln 2);
* an independent library (scipy.special.log_softmax for the eager entropy definition
  of the axolotl write-up, torch's float32 -> bfloat16 cast for the rounding routine);
* central finite differences of the forward for both backward passes;
* invariants (sum_j dlogits_j = 0, 0 <= H <= ln V, shift invariance, zero gradient
  exactly where clipping binds, +0.0 rows where the row gradient is zero).

``tests/test_oracle_pins.py`` runs them on the oracle; ``tests/test_oracle_mutations.py``
plants plausible mistakes in copies of the oracle and checks that each one is caught.
"""

from __future__ import annotations

import math

import numpy as np

try:
    import mpmath
except ImportError:  # without mpmath, long double stands in
    mpmath = None


def _close(a, b, rtol, atol, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    bad = ~(np.abs(a - b) <= atol + rtol * np.abs(b))
    assert not np.any(bad), f"{what}: max |diff| {np.max(np.abs(a - b))} (first bad {a[bad][:3]} vs {b[bad][:3]})"


# ---------------------------------------------------------------------------
# exact conversions
# ---------------------------------------------------------------------------

def check_bf16_decode_all_patterns(orc):
    """Every one of the 65536 bf16 patterns decodes to the value torch gives it."""
    import torch
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = orc.bf16_bits_to_fp64(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert np.all(same), "bf16 decode differs from torch"


def check_bf16_rounding_vs_torch(orc):
    """On float32-representable inputs, direct fp64->bf16 RNE equals torch's fp32->bf16 cast."""
    import torch
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-40, 39, 20000),
        rng.standard_normal(2000) * 1e-39,                    # subnormal range
        np.array([0.0, -0.0, np.inf, -np.inf, 3.3e38, -3.39e38, 1e-45, -1e-45]),
    ]).astype(np.float32)
    # include exact ties: bf16 value + half a unit
    tie = (np.arange(1, 4000, dtype=np.uint32) << np.uint32(16)) | np.uint32(0x8000)
    vals = np.concatenate([vals, tie.view(np.float32)])
    vals = vals[np.isfinite(vals.astype(np.float64)) | np.isinf(vals)]
    ours = orc.round_to_bf16_bits(vals.astype(np.float64))
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref), f"{np.sum(ours != ref)} patterns differ from torch"


def check_bf16_rounding_direct_cases(orc):
    """Cases that rounding through float32 would get wrong, and the range edges."""
    cases = [
        (1.0 + 2.0 ** -8 + 2.0 ** -30, 0x3F81),   # just above a tie: up (fp32 first would tie to 1.0)
        (1.0 + 2.0 ** -8, 0x3F80),                # exact tie, even is 1.0
        (1.0 + 3 * 2.0 ** -8, 0x3F82),            # exact tie, even is the upper neighbour
        (-(1.0 + 2.0 ** -8 + 2.0 ** -40), 0xBF81),
        (2.0 ** -134, 0x0000),                    # half the smallest subnormal: tie to 0
        (2.0 ** -134 * (1 + 2.0 ** -20), 0x0001),
        (1.5 * 2.0 ** -133, 0x0002),              # subnormal tie to even
        (2.0 ** -126, 0x0080),                    # smallest normal
        ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),   # largest finite
        ((2 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),   # tie above the largest finite: to even = inf
        ((2 - 2.0 ** -8 - 2.0 ** -30) * 2.0 ** 127, 0x7F7F),
        (1e300, 0x7F80), (-1e300, 0xFF80),
        (0.0, 0x0000), (-0.0, 0x8000), (np.inf, 0x7F80), (-np.inf, 0xFF80),
        (float("nan"), 0x7FC0),
    ]
    got = orc.round_to_bf16_bits(np.array([c[0] for c in cases]))
    for (v, want), g in zip(cases, got):
        assert int(g) == want, f"round_to_bf16_bits({v!r}) = {int(g):#06x}, want {want:#06x}"


# ---------------------------------------------------------------------------
# log-softmax, selective gather, entropy
# ---------------------------------------------------------------------------

def _brute_row(x, idx, T):
    """lse, logp, H of one row by high-precision arithmetic, no max shift."""
    if mpmath is not None:
        mpmath.mp.dps = 50
        z = [mpmath.mpf(float(v)) / mpmath.mpf(float(T)) for v in x]
        S = mpmath.fsum([mpmath.e ** zj for zj in z])
        lse = mpmath.log(S)
        p = [mpmath.e ** zj / S for zj in z]
        H = -mpmath.fsum([pj * mpmath.log(pj) for pj in p if pj > 0])
        return float(lse), float(z[idx] - lse), float(H)
    z = np.asarray(x, dtype=np.longdouble) / np.longdouble(T)
    S = np.sum(np.exp(z))
    lse = np.log(S)
    p = np.exp(z) / S
    H = -np.sum(p * np.log(p))
    return float(lse), float(z[idx] - lse), float(H)


def check_brute_force_tiny_rows(orc):
    """lse, logp and H against high-precision brute force (no shift) on tiny rows, T != 1."""
    rng = np.random.default_rng(2)
    for V in (1, 2, 3, 5, 8):
        for T in (1.0, 0.7, 1.9):
            x = rng.standard_normal((4, V)) * 3.0
            idx = rng.integers(0, V, 4)
            logp, lse = orc.selective_log_softmax(x, idx, T)
            H = orc.entropy_from_logits(x, T)
            for r in range(4):
                b_lse, b_logp, b_H = _brute_row(x[r], idx[r], T)
                _close(lse[r], b_lse, 1e-13, 1e-13, f"lse V={V} T={T}")
                _close(logp[r], b_logp, 1e-12, 1e-12, f"logp V={V} T={T}")
                _close(H[r], b_H, 1e-12, 1e-12, f"H V={V} T={T}")


def check_closed_form_v2(orc):
    """V = 2: logp_idx = -log(1 + exp(z_other - z_idx)); H of a Bernoulli."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((50, 2)) * 4.0
    idx = rng.integers(0, 2, 50)
    T = 1.3
    logp, lse = orc.selective_log_softmax(x, idx, T)
    zi = x[np.arange(50), idx] / T
    zo = x[np.arange(50), 1 - idx] / T
    _close(logp, -np.log1p(np.exp(zo - zi)), 1e-13, 1e-14, "V=2 logp")
    q = 1.0 / (1.0 + np.exp(zo - zi))
    H = orc.entropy_from_logits(x, T)
    _close(H, -(q * np.log(q) + (1 - q) * np.log(1 - q)), 1e-12, 1e-14, "V=2 entropy")


def check_uniform_and_two_level_rows(orc):
    """All-equal rows: lse = z + ln V, logp = -ln V, H = ln V.  Two-level rows: closed form."""
    for V in (1, 7, 512, 32000):
        x = np.full((3, V), 1.75)
        idx = np.array([0, V // 2, V - 1])
        logp, lse = orc.selective_log_softmax(x, idx, 0.5)
        _close(lse, 3.5 + math.log(V), 1e-13, 1e-13, "uniform lse")
        _close(logp, -math.log(V) * np.ones(3), 1e-12, 1e-13, "uniform logp")
        _close(orc.entropy_from_logits(x, 0.5), math.log(V) * np.ones(3), 1e-12, 1e-12, "uniform H")
    # k entries at level a, V-k at 0 (T = 1): p_hi = e^a / (k e^a + V - k)
    V, k, a = 1000, 3, 5.0
    x = np.zeros((1, V)); x[0, :k] = a
    Z = k * math.exp(a) + (V - k)
    ph, pl = math.exp(a) / Z, 1.0 / Z
    H_ref = -(k * ph * math.log(ph) + (V - k) * pl * math.log(pl))
    _close(orc.entropy_from_logits(x, 1.0), [H_ref], 1e-12, 1e-13, "two-level H")
    logp, _ = orc.selective_log_softmax(x, np.array([0]), 1.0)
    _close(logp, [math.log(ph)], 1e-13, 1e-13, "two-level logp")


def check_entropy_vs_scipy_eager_definition(orc):
    """H = -sum exp(log_softmax) * log_softmax (axolotl write-up, original implementation),
    evaluated with scipy's log_softmax."""
    from scipy.special import log_softmax
    rng = np.random.default_rng(4)
    x = rng.standard_normal((16, 3000)) * 3.0
    x[3, 17] += 20.0
    for T in (1.0, 0.7):
        ls = log_softmax(x / T, axis=-1)
        ref = -np.sum(np.exp(ls) * ls, axis=-1)
        _close(orc.entropy_from_logits(x, T), ref, 1e-11, 1e-12, "entropy vs scipy")
        logp, _ = orc.selective_log_softmax(x, np.arange(16) * 7, T)
        _close(logp, ls[np.arange(16), np.arange(16) * 7], 1e-12, 1e-12, "logp vs scipy")


def check_entropy_bounds_and_spike(orc):
    """0 <= H <= ln V on random rows; one huge spike gives H ~ 0 and logp ~ 0 at the spike."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((64, 777)) * rng.uniform(0.1, 10.0, (64, 1))
    H = orc.entropy_from_logits(x, 1.0)
    assert np.all(H >= 0.0) and np.all(H <= math.log(777) + 1e-12), "entropy out of [0, ln V]"
    y = np.zeros((1, 100)); y[0, 42] = 1000.0
    assert orc.entropy_from_logits(y, 1.0)[0] < 1e-300 + 1e-12
    logp, lse = orc.selective_log_softmax(y, np.array([42]), 1.0)
    _close(lse, [1000.0], 0, 1e-12, "spike lse (needs the max shift)")
    _close(logp, [0.0], 0, 1e-12, "spike logp")


def check_special_rows(orc):
    """An all -inf row: lse = log(0) = -inf, logp and H undefined (NaN).  A NaN logit makes
    the row NaN.  A -inf logit among finite ones contributes exp(-inf) = 0 to the sum and
    0 to the entropy."""
    x = np.array([[-np.inf] * 4, [0.0, np.nan, 1.0, 2.0], [0.0, -np.inf, 1.0, 2.0]])
    with np.errstate(all="ignore"):
        logp, lse = orc.selective_log_softmax(x, np.array([0, 0, 2]), 1.0)
        H = orc.entropy_from_logits(x, 1.0)
    assert np.isneginf(lse[0]) and np.isnan(logp[0]) and np.isnan(H[0])
    assert np.isnan(lse[1]) and np.isnan(logp[1]) and np.isnan(H[1])
    ref = math.log(1 + math.e + math.e ** 2)
    _close(lse[2:], [ref], 1e-14, 0, "lse with a -inf logit")
    _close(logp[2:], [1.0 - ref], 1e-14, 0, "logp with a -inf logit")
    # the -inf entry has p = 0 and adds nothing (p log p -> 0): H of the other three
    q = np.exp(np.array([0.0, 1.0, 2.0]) - ref)
    _close(H[2:], [-np.sum(q * np.log(q))], 1e-13, 0, "entropy with a -inf logit")


def check_shift_invariance(orc):
    """x + c leaves logp and H unchanged and shifts lse by c / T."""
    rng = np.random.default_rng(6)
    x = rng.standard_normal((8, 200)) * 2.0
    idx = rng.integers(0, 200, 8)
    T = 0.8
    lp0, lse0 = orc.selective_log_softmax(x, idx, T)
    lp1, lse1 = orc.selective_log_softmax(x + 37.0, idx, T)
    _close(lp1, lp0, 1e-11, 1e-11, "shift logp")
    _close(lse1, lse0 + 37.0 / T, 1e-13, 1e-11, "shift lse")
    _close(orc.entropy_from_logits(x + 37.0, T), orc.entropy_from_logits(x, T), 1e-10, 1e-11, "shift H")


# ---------------------------------------------------------------------------
# GRPO per-token terms: textbook cases of the clipped objective and the k3 KL
# ---------------------------------------------------------------------------

def _terms(orc, logp, old, ref, A, beta=0.0, el=0.2, eh=0.28, mask=None):
    logp = np.atleast_1d(np.asarray(logp, dtype=np.float64))
    n = logp.shape[0]
    old = None if old is None else np.broadcast_to(np.asarray(old, dtype=np.float64), (n,))
    ref = None if ref is None else np.broadcast_to(np.asarray(ref, dtype=np.float64), (n,))
    A = np.broadcast_to(np.asarray(A, dtype=np.float64), (n,))
    t = orc.grpo_token_terms(logp, old, ref, A, mask, beta, el, eh)
    d = orc.grpo_dlogp(logp, old, ref, A, mask, beta, el, eh)
    return t, d


def check_ppo_clip_textbook_cases(orc):
    """The six regions of the PPO clipped objective with asymmetric eps (0.2 low, 0.28 high)."""
    lp = -2.0
    cases = [
        # (log ratio, A, pg, clipped, dpg)
        (0.0, 1.5, -1.5, False, -1.5),                                # ratio 1
        (math.log(1.5), 2.0, -1.28 * 2.0, True, 0.0),                  # A>0, r>1+eh: clipped
        (math.log(0.5), 2.0, -0.5 * 2.0, False, -2.0 * 0.5),           # A>0, r<1-el: pessimistic r*A
        (math.log(0.5), -2.0, -0.8 * -2.0, True, 0.0),                 # A<0, r<1-el: clipped
        (math.log(1.5), -2.0, -1.5 * -2.0, False, 2.0 * 1.5),          # A<0, r>1+eh: r*A
        (math.log(1.1), 3.0, -1.1 * 3.0, False, -3.0 * 1.1),           # inside the range
        (math.log(0.9), -3.0, -0.9 * -3.0, False, 3.0 * 0.9),          # inside the range, A<0
        (math.log(1.2), 1.0, -1.2, False, -1.2),                       # between 1+el and 1+eh: not clipped
        (math.log(0.75), -1.0, 0.8, True, 0.0),                        # r < 1-el = 0.8 with A<0
    ]
    for lr, A, pg, clipped, dpg in cases:
        t, d = _terms(orc, [lp], [lp - lr], None, [A])
        _close(t["pg"], [pg], 1e-12, 1e-14, f"pg lr={lr} A={A}")
        _close(t["loss"], [pg], 1e-12, 1e-14, f"loss lr={lr} A={A}")
        assert bool(t["is_clipped"][0]) == clipped, f"is_clipped lr={lr} A={A}"
        _close(d, [dpg], 1e-12, 1e-14, f"dlogp lr={lr} A={A}")
        _close(t["ratio"], [math.exp(lr)], 1e-14, 0, "ratio")


def check_clip_boundary_ties(orc):
    """A ratio exactly on a clip boundary is not clipped and keeps the -A*r gradient
    (both branches of the min have that derivative there)."""
    for r, A in ((1.25, 2.0), (0.75, -2.0)):
        # eps chosen so that 1 + eh == r and 1 - el == r exactly in binary
        t = orc.grpo_token_terms(np.array([0.0]), np.array([-math.log(r)]), None, np.array([A]), None,
                                 0.0, 0.25, 0.25)
        ratio = float(t["ratio"][0])
        # use the oracle's own fp64 ratio as the boundary so the tie is exact
        el = eh = abs(ratio - 1.0)
        t = orc.grpo_token_terms(np.array([0.0]), np.array([-math.log(r)]), None, np.array([A]), None, 0.0, el, eh)
        d = orc.grpo_dlogp(np.array([0.0]), np.array([-math.log(r)]), None, np.array([A]), None, 0.0, el, eh)
        assert not bool(t["is_clipped"][0]), "tie counted as clipped"
        _close(d, [-A * ratio], 1e-14, 0, "tie gradient")


def check_zero_advantage_and_mask(orc):
    """A == 0 gives pg = 0, no clipping and (with beta == 0) a zero row gradient;
    masked tokens give +0.0 for every output and a zero gradient."""
    t, d = _terms(orc, [-1.0, -2.0], [-1.5, -0.3], None, [0.0, 0.0])
    assert np.all(t["pg"] == 0.0) and not np.any(t["is_clipped"]) and np.all(d == 0.0)
    mask = np.array([1, 0, 0], dtype=np.uint8)
    t, d = _terms(orc, [-1.0, -2.0, -3.0], [-1.2, -2.5, -3.0], [-1.1, -1.0, -2.0], [1.0, -1.0, 2.0],
                  beta=0.1, mask=mask)
    for k in ("pg", "kl", "loss"):
        assert np.all(t[k][1:] == 0.0) and not np.any(np.signbit(t[k][1:])), f"masked {k} not +0"
    assert not np.any(t["is_clipped"][1:])
    assert np.all(d[1:] == 0.0)
    assert t["loss"][0] != 0.0 and d[0] != 0.0


def check_k3_kl_closed_forms(orc):
    """kl = beta (e^d - d - 1) at d = ref - logp in {0, ln 2, -ln 2}; its gradient is the
    expression the Liger write-up prints, beta * (1 - exp(ref_logp - logp))."""
    beta = 0.04
    lp = np.array([-1.0, -1.0, -1.0])
    ref = lp + np.array([0.0, math.log(2.0), -math.log(2.0)])
    t, d = _terms(orc, lp, None, ref, [0.0, 0.0, 0.0], beta=beta)
    _close(t["kl"], [0.0, beta * (1 - math.log(2)), beta * (math.log(2) - 0.5)], 1e-13, 1e-16, "kl")
    _close(d, [0.0, -beta, beta * 0.5], 1e-13, 1e-16, "dkl")
    assert t["kl"][0] == 0.0 and d[0] == 0.0
    # beta == 0 never evaluates the KL term (ref may even be absent)
    t, d = _terms(orc, lp, None, None, [0.0, 0.0, 0.0], beta=0.0)
    assert np.all(t["kl"] == 0.0) and np.all(d == 0.0)


# ---------------------------------------------------------------------------
# backward: finite differences, invariants, zero rows
# ---------------------------------------------------------------------------

def _fd_problem(seed=7, B=2, L=6, V=13):
    rng = np.random.default_rng(seed)
    R = B * L
    x = rng.standard_normal((R, V)) * 2.0
    idx = rng.integers(0, V, R)
    A = rng.standard_normal(B)
    return rng, x, idx, A


def check_grpo_bwd_finite_differences(orc):
    """dlogits of J = sum_r dloss_r * loss_r(x) against central differences of the forward,
    with T != 1, beta > 0, asymmetric eps, a mask, and rows far from a clip boundary."""
    rng, x, idx, A = _fd_problem()
    R, V = x.shape
    L = 6
    T, beta, el, eh = 0.7, 0.1, 0.2, 0.28
    adv = orc.per_row(A, L)
    logp0, _ = orc.selective_log_softmax(x, idx, T)
    old = logp0 + rng.standard_normal(R) * 0.3
    ref = logp0 + rng.standard_normal(R) * 0.2
    mask = (rng.uniform(size=R) > 0.2).astype(np.uint8)
    dloss = rng.uniform(0.1, 1.0, R)
    r = np.exp(logp0 - old)
    far = (np.abs(r - (1 - el)) > 0.02) & (np.abs(r - (1 + eh)) > 0.02)
    dl, g = orc.grpo_loss_bwd(x, idx, old, ref, adv, mask, dloss, T, beta, el, eh)

    def J_rows(xx):
        out = orc.grpo_loss_fwd(xx, idx_rep, old_rep, ref_rep, adv_rep, mask_rep, T, beta, el, eh)
        return out["loss"] * dloss_rep

    h = 1e-6
    for rr in np.nonzero(far)[0]:
        # perturb every column of row rr at once: V copies of the row
        xp = np.repeat(x[rr:rr + 1], V, axis=0) + h * np.eye(V)
        xm = np.repeat(x[rr:rr + 1], V, axis=0) - h * np.eye(V)
        idx_rep = np.full(V, idx[rr]); old_rep = np.full(V, old[rr]); ref_rep = np.full(V, ref[rr])
        adv_rep = np.full(V, adv[rr]); mask_rep = np.full(V, mask[rr]); dloss_rep = np.full(V, dloss[rr])
        fd = (J_rows(xp) - J_rows(xm)) / (2 * h)
        _close(dl[rr], fd, 1e-6, 1e-9, f"grpo dlogits row {rr}")
    assert np.sum(far & (mask == 1)) >= 5, "finite-difference problem has too few live rows"


def check_slsm_bwd_finite_differences(orc):
    """dlogits of J = sum_r u_r * logp_r(x) against central differences, T != 1."""
    rng, x, idx, _ = _fd_problem(seed=8)
    R, V = x.shape
    T = 1.6
    u = rng.standard_normal(R)
    dl, _ = orc.selective_log_softmax_bwd(x, idx, u, T)
    h = 1e-6
    for rr in range(R):
        xp = np.repeat(x[rr:rr + 1], V, axis=0) + h * np.eye(V)
        xm = np.repeat(x[rr:rr + 1], V, axis=0) - h * np.eye(V)
        fp, _ = orc.selective_log_softmax(xp, np.full(V, idx[rr]), T)
        fm, _ = orc.selective_log_softmax(xm, np.full(V, idx[rr]), T)
        _close(dl[rr], u[rr] * (fp - fm) / (2 * h), 1e-6, 1e-9, f"slsm dlogits row {rr}")


def check_bwd_invariants(orc):
    """sum_j dlogits_j = 0 per row; zero gradient exactly where clipping binds (beta = 0);
    rows with a zero row gradient are +0.0 bits, including when it is -0.0."""
    rng = np.random.default_rng(9)
    B, L, V = 3, 40, 64
    R = B * L
    x = rng.standard_normal((R, V)) * 2.0
    idx = rng.integers(0, V, R)
    A = np.array([0.7, 0.0, -1.3])
    adv = orc.per_row(A, L)
    T = 0.9
    logp0, _ = orc.selective_log_softmax(x, idx, T)
    old = logp0 + rng.standard_normal(R) * 0.4
    mask = (np.arange(R) % L < 35).astype(np.uint8)
    dloss = mask / 35.0
    dl, g = orc.grpo_loss_bwd(x, idx, old, None, adv, mask, dloss, T, 0.0, 0.2, 0.2)
    sums = dl.sum(axis=1)
    assert np.all(np.abs(sums) <= 1e-12 * np.maximum(np.abs(g), 1e-300) + 1e-300), "row sums not 0"
    t = orc.grpo_token_terms(logp0, old, None, adv, mask, 0.0, 0.2, 0.2)
    live = (mask == 1) & (adv != 0.0)
    assert np.array_equal(g[live] == 0.0, t["is_clipped"][live]), "zero gradient != clipping binds"
    assert np.any(t["is_clipped"][live]) and np.any(~t["is_clipped"][live])
    zero_rows = g == 0.0
    assert np.any(zero_rows & (adv == 0.0)) and np.any(zero_rows & (mask == 0))
    assert np.all(dl[zero_rows] == 0.0) and not np.any(np.signbit(dl[zero_rows])), "zero rows not +0.0"
    # an upstream -0.0 gives a +0.0 row as well
    dl2, _ = orc.selective_log_softmax_bwd(x[:2], idx[:2], np.array([-0.0, 0.0]), T)
    assert np.all(dl2 == 0.0) and not np.any(np.signbit(dl2)), "-0.0 upstream row not +0.0"


def check_bwd_closed_form_on_policy(orc):
    """old = logp (ratio 1), beta = 0: dlogits = -A * dloss / T * (onehot - softmax)."""
    rng = np.random.default_rng(10)
    R, V, T = 6, 50, 0.8
    x = rng.standard_normal((R, V))
    idx = rng.integers(0, V, R)
    adv = rng.standard_normal(R)
    dloss = rng.uniform(0.5, 2.0, R)
    dl, _ = orc.grpo_loss_bwd(x, idx, None, None, adv, None, dloss, T, 0.0, 0.2, 0.2)
    from scipy.special import softmax
    p = softmax(x / T, axis=-1)
    onehot = np.eye(V)[idx]
    _close(dl, (-adv * dloss / T)[:, None] * (onehot - p), 1e-12, 1e-15, "on-policy closed form")


def check_entropy_bwd_finite_differences(orc):
    """dlogits of J = sum_r u_r * H_r(x) against central differences, T != 1; rows sum to 0;
    u = 0 rows are +0.0."""
    rng, x, idx, _ = _fd_problem(seed=11, V=17)
    R, V = x.shape
    T = 0.6
    u = rng.standard_normal(R)
    u[2] = 0.0
    dl, g = orc.entropy_from_logits_bwd(x, u, T)
    h = 1e-6
    for rr in range(R):
        xp = np.repeat(x[rr:rr + 1], V, axis=0) + h * np.eye(V)
        xm = np.repeat(x[rr:rr + 1], V, axis=0) - h * np.eye(V)
        fd = u[rr] * (orc.entropy_from_logits(xp, T) - orc.entropy_from_logits(xm, T)) / (2 * h)
        _close(dl[rr], fd, 1e-6, 1e-9, f"entropy dlogits row {rr}")
    assert np.all(np.abs(dl.sum(axis=1)) <= 1e-12 * (1 + np.abs(g)))
    assert np.all(dl[2] == 0.0) and not np.any(np.signbit(dl[2]))


def check_entropy_bwd_closed_form_v2(orc):
    """V = 2, T = 1: H(q) of a Bernoulli with q = sigmoid(x0 - x1); dH/dx0 = q(1-q) log((1-q)/q)."""
    rng = np.random.default_rng(12)
    x = rng.standard_normal((20, 2)) * 3.0
    dl, _ = orc.entropy_from_logits_bwd(x, np.ones(20), 1.0)
    q = 1.0 / (1.0 + np.exp(x[:, 1] - x[:, 0]))
    ref0 = q * (1 - q) * np.log((1 - q) / q)
    _close(dl[:, 0], ref0, 1e-11, 1e-14, "V=2 entropy gradient")
    _close(dl[:, 1], -ref0, 1e-11, 1e-14, "V=2 entropy gradient (other column)")


def check_seq_bwd_finite_differences(orc):
    """Sequence-level objective J = sum_t dloss_t loss_t(x): its dlogits against central
    differences over every logit of every sequence (the sequence ratio couples the rows)."""
    rng = np.random.default_rng(13)
    B, L, V = 2, 4, 7
    R = B * L
    x = rng.standard_normal((R, V)) * 1.5
    idx = rng.integers(0, V, R)
    A = np.array([0.9, -1.4])
    T, beta, el, eh = 0.8, 0.07, 0.2, 0.28
    lp0, _ = orc.selective_log_softmax(x, idx, T)
    old = lp0 + rng.standard_normal(R) * 0.05
    ref = lp0 + rng.standard_normal(R) * 0.2
    mask = np.array([1, 1, 1, 0, 1, 1, 0, 0], dtype=np.uint8)
    dloss = rng.uniform(0.2, 1.0, R) * mask
    dl, g, terms = orc.grpo_seq_loss_bwd(x, idx, old, ref, A, mask, dloss, B, L, T, beta, el, eh)
    s = terms["seq_ratio"]
    assert np.all(np.abs(s - (1 - el)) > 0.02) and np.all(np.abs(s - (1 + eh)) > 0.02)

    def J(xx):
        lp, _ = orc.selective_log_softmax(xx, idx, T)
        t = orc.grpo_seq_terms(lp, old, ref, A, mask, dloss, B, L, beta, el, eh)
        return float(np.sum(dloss * t["loss"]))

    h = 1e-6
    fd = np.zeros((R, V))
    for r in range(R):
        for j in range(V):
            xp = x.copy(); xp[r, j] += h
            xm = x.copy(); xm[r, j] -= h
            fd[r, j] = (J(xp) - J(xm)) / (2 * h)
    _close(dl, fd, 1e-6, 1e-9, "sequence-level dlogits")
    assert np.all(dl[mask == 0] == 0.0)


def check_seq_terms_closed_forms(orc):
    """old = logp: s = 1, pg = -A, dpg/dlogp_t = -A / n; a clipped sequence (A > 0, s > 1 + eps)
    has a zero policy gradient; a sequence without tokens has ratio 1 and zero terms."""
    B, L = 3, 4
    lp = np.linspace(-3.0, -1.0, B * L)
    mask = np.array([1, 1, 1, 1, 1, 1, 0, 0, 0, 0, 0, 0], dtype=np.uint8)
    dloss = mask / 4.0
    A = np.array([2.0, 1.0, 5.0])
    old = lp.copy()
    old[4:6] = lp[4:6] - 1.0                    # sequence 1: s = e (> 1 + eps_high)
    t = orc.grpo_seq_terms(lp, old, None, A, mask, dloss, B, L, 0.0, 0.2, 0.28)
    _close(t["seq_ratio"], [1.0, math.e, 1.0], 1e-14, 0, "seq ratio")
    _close(t["seq_pg"][:2], [-2.0, -1.28 * 1.0], 1e-14, 0, "seq pg")
    assert list(t["seq_is_clipped"]) == [False, True, False]
    W0 = 1.0                                     # sum of dloss over sequence 0
    _close(t["dlogp"][:4], np.full(4, W0 * -2.0 * 1.0 / 4), 1e-14, 0, "seq dlogp, on-policy")
    assert np.all(t["dlogp"][4:] == 0.0) and np.all(t["loss"][8:] == 0.0)


# ---------------------------------------------------------------------------
# the GRPO loss on top of the LM head (hidden states and head weight)
# ---------------------------------------------------------------------------

def _linear_problem(seed=11, B=2, L=5, H=7, V=13):
    rng = np.random.default_rng(seed)
    R = B * L
    h = rng.standard_normal((R, H))
    W = rng.standard_normal((V, H)) * 0.7
    idx = rng.integers(0, V, R)
    A = rng.standard_normal(B)
    return rng, h, W, idx, A


def check_fused_linear_finite_differences(orc):
    """grad_h and grad_W of J = sum_r dloss_r * loss_r(h W^T) against central differences
    in every element of h and of W (beta > 0, T != 1, asymmetric eps, a mask)."""
    rng, h, W, idx, A = _linear_problem()
    R, H = h.shape
    V = W.shape[0]
    L = 5
    T, beta, el, eh = 0.8, 0.07, 0.2, 0.28
    adv = orc.per_row(A, L)
    lp0, _ = orc.selective_log_softmax(h @ W.T, idx, T)
    old = lp0 + rng.standard_normal(R) * 0.25
    ref = lp0 + rng.standard_normal(R) * 0.15
    mask = np.ones(R, np.uint8)
    mask[[2, 7]] = 0
    dloss = rng.uniform(0.1, 1.0, R)
    r = np.exp(lp0 - old)
    assert np.all((np.abs(r - (1 - el)) > 0.01) & (np.abs(r - (1 + eh)) > 0.01)), "a row sits on a clip boundary"
    _, gh, gW, _ = orc.fused_linear_grpo(h, W, idx, old, ref, adv, mask, dloss, T, beta, el, eh)

    def J(hh, WW):
        f = orc.grpo_loss_fwd(hh @ WW.T, idx, old, ref, adv, mask, T, beta, el, eh)
        return float(np.sum(f["loss"] * dloss))

    eps = 1e-6
    fd_h = np.zeros_like(h)
    for i in range(R):
        for k in range(H):
            e = np.zeros_like(h)
            e[i, k] = eps
            fd_h[i, k] = (J(h + e, W) - J(h - e, W)) / (2 * eps)
    fd_W = np.zeros_like(W)
    for j in range(V):
        for k in range(H):
            e = np.zeros_like(W)
            e[j, k] = eps
            fd_W[j, k] = (J(h, W + e) - J(h, W - e)) / (2 * eps)
    _close(gh, fd_h, 1e-6, 1e-9, "grad_h")
    _close(gW, fd_W, 1e-6, 1e-9, "grad_W")
    assert np.all(gh[[2, 7]] == 0.0), "masked rows get no hidden-state gradient"


def check_fused_linear_identity_head_and_invariants(orc):
    """A head W = s I (H = V) gives the row pass on x = s h: the same forward, grad_h =
    s dx.  A head whose rows are all equal gives uniform p and grad_h = 0 (each row of dx
    sums to 0); every column of grad_W sums to 0 over the vocabulary for any head."""
    rng, h, _, idx, A = _linear_problem(seed=12, H=9, V=9)
    R, H = h.shape
    L = 5
    T, beta, el, eh = 1.3, 0.0, 0.2, 0.2
    adv = orc.per_row(A, L)
    old = rng.standard_normal(R) * 0.1 - 2.0
    dloss = rng.uniform(0.2, 1.0, R)
    s = 1.7
    f, gh, gW, dx = orc.fused_linear_grpo(h, s * np.eye(H), idx, old, None, adv, None, dloss, T, beta, el, eh)
    f2 = orc.grpo_loss_fwd(s * h, idx, old, None, adv, None, T, beta, el, eh)
    d2, _ = orc.grpo_loss_bwd(s * h, idx, old, None, adv, None, dloss, T, beta, el, eh)
    for k in ("loss", "logp", "lse", "entropy"):
        _close(f[k], f2[k], 1e-13, 1e-13, f"identity head {k}")
    _close(gh, s * d2, 1e-12, 1e-14, "identity head grad_h")
    w = rng.standard_normal(H)
    _, gh_eq, gW_eq, _ = orc.fused_linear_grpo(h, np.tile(w, (11, 1)), idx % 11, old, None, adv, None, dloss, T,
                                               beta, el, eh)
    _close(gh_eq, np.zeros_like(gh_eq), 0, 1e-12, "equal head rows: grad_h = 0")
    for g in (gW, gW_eq):
        _close(g.sum(axis=0), np.zeros(H), 0, 1e-12, "grad_W columns sum to 0")


ALL_CHECKS = [
    check_bf16_decode_all_patterns,
    check_bf16_rounding_vs_torch,
    check_bf16_rounding_direct_cases,
    check_brute_force_tiny_rows,
    check_closed_form_v2,
    check_uniform_and_two_level_rows,
    check_entropy_vs_scipy_eager_definition,
    check_entropy_bounds_and_spike,
    check_special_rows,
    check_shift_invariance,
    check_ppo_clip_textbook_cases,
    check_clip_boundary_ties,
    check_zero_advantage_and_mask,
    check_k3_kl_closed_forms,
    check_grpo_bwd_finite_differences,
    check_slsm_bwd_finite_differences,
    check_bwd_invariants,
    check_bwd_closed_form_on_policy,
    check_entropy_bwd_finite_differences,
    check_entropy_bwd_closed_form_v2,
    check_seq_bwd_finite_differences,
    check_seq_terms_closed_forms,
    check_fused_linear_finite_differences,
    check_fused_linear_identity_head_and_invariants,
]
