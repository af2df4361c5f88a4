"""fp64 CPU oracle for the GRPO / entropy / selective-log-softmax row pass.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, obviously correct
definition of what the CUDA library computes.  Only the test suite, the smoke
check in ``__graft_entry__.smoke`` and the ``cpu_baseline`` / reference leg of
``bench.py`` may import it.  The product path (the C-ABI library and its Python
binding) never calls it, and it shares no code with that path: no kernels, no
helpers, no constants, no pre- or post-processing.

Sources (the three web pages the method is described on):

* [Liger-bwd]  "LinkedIn Liger-Kernel GRPO Loss Backward optimisation: 50%
  faster by removing needless work" (write-up of Liger-Kernel PR #1550).
  Sections used: "Code analysis" (the ``_grpo_loss_bwd_kernel`` and
  ``_grpo_loss_bwd_kernel_seq`` diffs), "Why it's good", "Review feedback
  analysis".
* [Liger-TRL]  "Liger GRPO meets TRL".  Sections used: "2. The core principle
  that sets GRPO apart from PPO" (group-relative, verifiable rewards),
  "3. The memory bottleneck of storing the full logits" (the logits are the LM head
  applied to the hidden states), "4. The chunked loss that computes gradients during
  the forward".
* [axolotl]    "Axolotl: entropy and selective log-softmax with Triton kernels"
  (write-up of axolotl PR #3510).  Sections used: "1. benchmarks/bench_entropy.py"
  (the original eager entropy definition), "2. benchmarks/bench_selective_logsoftmax.py".

Notation (one row r = one token (b, l) of a [B, L, V] logits tensor):

* x_j     raw logit, j in [0, V); decoded exactly from bf16 or fp32 bits
* T       sampling temperature; z_j = x_j / T
* lse     log sum_j exp(z_j)
* p_j     exp(z_j - lse)
* idx     the sampled token of the row; logp = z_idx - lse
* H       entropy  -sum_j p_j log p_j  =  sum_j p_j (lse - z_j)

Parity status per function: every public function below is pinned by
``tests/test_oracle_pins.py`` against brute force (mpmath / long double),
closed forms, an independent library (scipy), finite differences or an
invariant.  None is "parity unpinned".
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "decode_logits",
    "round_to_bf16_bits",
    "round_to_fp32",
    "bf16_bits_to_fp64",
    "log_softmax_rows",
    "selective_log_softmax",
    "entropy_from_logits",
    "grpo_token_terms",
    "grpo_dlogp",
    "softmax_gather_grad",
    "grpo_loss_fwd",
    "grpo_loss_bwd",
    "selective_log_softmax_bwd",
    "entropy_from_logits_bwd",
    "grpo_seq_terms",
    "grpo_seq_loss_bwd",
    "fused_linear_grpo",
    "per_row",
]


# ---------------------------------------------------------------------------
# exact conversions
# ---------------------------------------------------------------------------

def bf16_bits_to_fp64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly.

    A bf16 value is the upper half of an IEEE binary32 pattern, so shifting the
    16 bits into the top of a 32-bit word and reading it as float32 gives the
    value exactly; float32 -> float64 is exact as well.
    """
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def decode_logits(raw, dtype: str) -> np.ndarray:
    """Raw logits as stored ('bf16': uint16 bit patterns, 'fp32': float32) -> float64."""
    if dtype == "bf16":
        return bf16_bits_to_fp64(raw)
    if dtype == "fp32":
        return np.asarray(raw, dtype=np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


_BF16_MANT_BITS = 7          # stored mantissa bits of bf16
_BF16_MIN_EXP = -126         # exponent of the smallest normal bf16 (same as binary32)


def round_to_bf16_bits(v) -> np.ndarray:
    """Round float64 values to bf16 with round-to-nearest-even, DIRECTLY.

    Rounding through float32 first would round twice; this routine instead
    scales |v| so that one unit of the bf16 grid at |v| becomes 1.0, rounds to
    the nearest integer with ties to even (``np.rint``), and scales back.  All
    scalings are by powers of two and therefore exact.  The grid spacing is
    2**(e - 7) for a normal value in [2**e, 2**(e+1)) and 2**-133 in the
    subnormal range.  Results beyond the largest finite bf16 become +-inf, NaN
    becomes the canonical quiet NaN 0x7FC0 (sign kept), and the sign of zero is
    kept.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    with np.errstate(over="ignore", invalid="ignore"):
        a = np.abs(v)
        _, e = np.frexp(a)                      # a = f * 2**e with f in [0.5, 1)
        # exponent of one grid unit at a: (e - 1) - 7, floored at the subnormal unit
        unit_exp = np.maximum(e - 1 - _BF16_MANT_BITS, _BF16_MIN_EXP - _BF16_MANT_BITS)
        q = np.rint(np.ldexp(a, -unit_exp))     # exact scaling, then RNE to an integer
        r = np.ldexp(q, unit_exp)               # back on the bf16 grid (exact)
        r32 = np.copysign(r, v).astype(np.float32)  # exact: every bf16 value is a float32 value
        bits = (r32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(v)
    if np.any(nan):
        sign = (np.signbit(v[nan]).astype(np.uint16) << np.uint16(15))
        bits[nan] = np.uint16(0x7FC0) | sign
    out[...] = bits
    return out


def round_to_fp32(v) -> np.ndarray:
    """Round float64 to float32 (IEEE round-to-nearest-even, as numpy's cast does)."""
    with np.errstate(over="ignore"):
        return np.asarray(v, dtype=np.float64).astype(np.float32)


def per_row(values_per_sequence, L: int) -> np.ndarray:
    """Broadcast a per-sequence array [B] to the B*L token rows (row r = b*L + l)."""
    return np.repeat(np.asarray(values_per_sequence, dtype=np.float64), L)


# ---------------------------------------------------------------------------
# row statistics: temperature-scaled log-softmax, selective gather, entropy
# ---------------------------------------------------------------------------

def log_softmax_rows(x: np.ndarray, T: float):
    """z = x / T and lse = log sum_j exp(z_j) for every row of x [n, V] (fp64).

    The temperature divides the logits before the softmax; [Liger-bwd], "Code
    analysis", divides the per-row gradient by the same TEMPERATURE, which is
    the chain-rule image of this scaling.  The sum is shifted by the row
    maximum so that exp never overflows; the shift cancels exactly in exact
    arithmetic.  A row whose logits are all -inf has an empty sum: lse = log 0
    = -inf (the shift is then 0, since -inf - (-inf) has no value).
    """
    x = np.asarray(x, dtype=np.float64)
    z = x / np.float64(T)
    with np.errstate(invalid="ignore", over="ignore", divide="ignore"):
        m = np.max(z, axis=-1, keepdims=True)
        m = np.where(np.isneginf(m), 0.0, m)
        s = np.sum(np.exp(z - m), axis=-1, keepdims=True)
        lse = (m + np.log(s))[..., 0]
    return z, lse


def selective_log_softmax(x: np.ndarray, idx: np.ndarray, T: float):
    """logp_r = log_softmax(x_r / T)[idx_r]; also returns lse_r.

    [axolotl], "2. benchmarks/bench_selective_logsoftmax.py": the operation
    evaluates the log-softmax only at the given index of each row.
    """
    z, lse = log_softmax_rows(x, T)
    rows = np.arange(z.shape[0])
    logp = z[rows, np.asarray(idx, dtype=np.int64)] - lse
    return logp, lse


def entropy_from_logits(x: np.ndarray, T: float = 1.0) -> np.ndarray:
    """H_r = sum_j p_j (lse - z_j)  (= -sum_j p_j log p_j), per row.

    [axolotl], "1. benchmarks/bench_entropy.py": the original implementation
    takes ``log_softmax`` of each row and returns minus the sum of
    ``exp(logps) * logps``.  Written here as sum_j p_j (lse - z_j) so every
    term is non-negative; the two are the same sum term by term.  The page's
    eager version has no temperature; T = 1 reproduces it.  A term with p_j = 0
    (a -inf logit, e.g. a vocabulary entry masked out) contributes 0, the limit
    of p log p as p -> 0.
    """
    z, lse = log_softmax_rows(x, T)
    with np.errstate(invalid="ignore"):
        p = np.exp(z - lse[:, None])
        return np.sum(np.where(p == 0.0, 0.0, p * (lse[:, None] - z)), axis=-1)


# ---------------------------------------------------------------------------
# GRPO per-token loss and its gradient with respect to logp
# ---------------------------------------------------------------------------

def grpo_token_terms(logp, old_logp, ref_logp, adv_row, mask, beta, eps_low, eps_high):
    """Per-token GRPO loss terms from logp (fp64).

    ratio  = exp(logp - old_logp)                       (old_logp None => ratio 1)
    pg     = -min(ratio * A, clip(ratio, 1 - eps_low, 1 + eps_high) * A)
    kl     = beta * (exp(ref - logp) - (ref - logp) - 1)   (beta == 0 => 0)
    loss   = pg + kl, and every output is +0.0 on a masked token.

    The pages print the gradient of the KL term, beta * (1 - exp(ref_logp -
    logp)) ([Liger-bwd], "Code analysis", both kernel diffs); the value above
    is the estimator whose derivative with respect to logp is exactly that.
    The clipped ratio objective is the PPO clip that [Liger-bwd], "Why it's
    good", names as the source of zero-gradient ("PPO-clipped") tokens; eps is
    taken asymmetric (eps_low, eps_high).  is_clipped marks tokens where the
    clipped branch is strictly the smaller one, i.e. where the policy-gradient
    term has zero gradient.
    """
    logp = np.asarray(logp, dtype=np.float64)
    n = logp.shape[0]
    A = np.asarray(adv_row, dtype=np.float64)
    mask = np.ones(n, dtype=bool) if mask is None else (np.asarray(mask) != 0)
    with np.errstate(over="ignore", invalid="ignore"):
        if old_logp is None:
            ratio = np.ones(n)
        else:
            ratio = np.exp(logp - np.asarray(old_logp, dtype=np.float64))
        clipped = np.clip(ratio, 1.0 - eps_low, 1.0 + eps_high)
        obj_unclipped = ratio * A
        obj_clipped = clipped * A
        pg = -np.minimum(obj_unclipped, obj_clipped)
        is_clipped = obj_clipped < obj_unclipped
        if beta != 0.0:
            d = np.asarray(ref_logp, dtype=np.float64) - logp
            kl = beta * (np.expm1(d) - d)          # exp(d) - d - 1 without cancellation
        else:
            kl = np.zeros(n)
        loss = pg + kl
    z = np.zeros(n)
    return {
        "ratio": ratio,
        "pg": np.where(mask, pg, z),
        "kl": np.where(mask, kl, z),
        "loss": np.where(mask, loss, z),
        "is_clipped": np.where(mask, is_clipped, False),
    }


def grpo_dlogp(logp, old_logp, ref_logp, adv_row, mask, beta, eps_low, eps_high):
    """d loss / d logp per token (fp64); 0 on masked tokens.

    Policy-gradient part: -A * ratio where the unclipped branch is the minimum
    (ties included: inside the clip range both branches have that derivative),
    0 where the clipped branch is strictly smaller (the clipped ratio is then
    constant in logp).  KL part: beta * (1 - exp(ref_logp - logp)), the term
    printed in [Liger-bwd], "Code analysis"; omitted when beta == 0.
    """
    logp = np.asarray(logp, dtype=np.float64)
    n = logp.shape[0]
    A = np.asarray(adv_row, dtype=np.float64)
    mask = np.ones(n, dtype=bool) if mask is None else (np.asarray(mask) != 0)
    with np.errstate(over="ignore", invalid="ignore"):
        if old_logp is None:
            ratio = np.ones(n)
        else:
            ratio = np.exp(logp - np.asarray(old_logp, dtype=np.float64))
        clipped = np.clip(ratio, 1.0 - eps_low, 1.0 + eps_high)
        unclipped_binds = (ratio * A) <= (clipped * A)
        dpg = np.where(unclipped_binds, -A * ratio, 0.0)
        if beta != 0.0:
            dkl = beta * (1.0 - np.exp(np.asarray(ref_logp, dtype=np.float64) - logp))
        else:
            dkl = np.zeros(n)
        dlogp = dpg + dkl
    return np.where(mask, dlogp, 0.0)


def softmax_gather_grad(x: np.ndarray, idx: np.ndarray, g: np.ndarray, T: float) -> np.ndarray:
    """dlogits_j = g * (1[j == idx] - p_j) per row, with rows where g == 0 all +0.0.

    g is the per-row factor (d loss / d logp) * (upstream) / T: d logp / d x_j
    = (1[j == idx] - p_j) / T.  A row whose g is exactly zero (either sign) is
    stored as +0.0 everywhere: [Liger-bwd], "Code analysis", adds an early
    return that stores 0.0 over the whole DLOGITS row when dlogp == 0.0, and
    "Why it's good" states outputs and gradients stay identical.
    """
    z, lse = log_softmax_rows(x, T)
    n, V = z.shape
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(invalid="ignore", over="ignore"):
        p = np.exp(z - lse[:, None])
        onehot = np.zeros((n, V))
        rows = np.arange(n)
        idx = np.asarray(idx, dtype=np.int64)
        ok = (idx >= 0) & (idx < V)
        onehot[rows[ok], idx[ok]] = 1.0
        d = g[:, None] * (onehot - p)
    d[g == 0.0, :] = 0.0                      # +0.0 bits (also for g == -0.0)
    return d


def grpo_loss_fwd(x, idx, old_logp, ref_logp, adv_row, mask, T, beta, eps_low, eps_high):
    """Forward of the GRPO row pass for rows x [n, V] (fp64).

    Returns loss, logp, lse, kl, is_clipped and entropy per row.  Masked rows
    have every output equal to +0.0 (and is_clipped False): their logits are
    not part of the objective.
    """
    n = np.asarray(x).shape[0]
    mask_b = np.ones(n, dtype=bool) if mask is None else (np.asarray(mask) != 0)
    logp, lse = selective_log_softmax(x, np.where(mask_b, idx, 0), T)
    H = entropy_from_logits(x, T)
    terms = grpo_token_terms(logp, old_logp, ref_logp, adv_row, mask_b, beta, eps_low, eps_high)
    z = np.zeros(n)
    return {
        "loss": terms["loss"],
        "logp": np.where(mask_b, logp, z),
        "lse": np.where(mask_b, lse, z),
        "kl": terms["kl"],
        "is_clipped": terms["is_clipped"],
        "entropy": np.where(mask_b, H, z),
        "ratio": terms["ratio"],
    }


def grpo_loss_bwd(x, idx, old_logp, ref_logp, adv_row, mask, dloss, T, beta, eps_low, eps_high):
    """Backward of sum_r dloss_r * loss_r with respect to the logits (fp64).

    g_r = dlogp_r * dloss_r / T ([Liger-bwd], "Code analysis":
    ``dlogp * dloss / TEMPERATURE``); dlogits_r = g_r * (onehot(idx_r) - p_r);
    rows with g_r == 0 are +0.0.  Returns (dlogits, g).
    """
    n = np.asarray(x).shape[0]
    mask_b = np.ones(n, dtype=bool) if mask is None else (np.asarray(mask) != 0)
    safe_idx = np.where(mask_b, idx, 0)
    logp, _ = selective_log_softmax(x, safe_idx, T)
    dlogp = grpo_dlogp(logp, old_logp, ref_logp, adv_row, mask_b, beta, eps_low, eps_high)
    g = dlogp * np.asarray(dloss, dtype=np.float64) / np.float64(T)
    g = np.where(mask_b, g, 0.0)
    return softmax_gather_grad(x, safe_idx, g, T), g


def selective_log_softmax_bwd(x, idx, dlogp_upstream, T):
    """Gradient of sum_r u_r * logp_r with respect to the logits (fp64).

    [axolotl], "2. benchmarks/bench_selective_logsoftmax.py": the backward of
    the selective log-softmax.  g_r = u_r / T; rows with g_r == 0 are +0.0.
    Returns (dlogits, g).
    """
    g = np.asarray(dlogp_upstream, dtype=np.float64) / np.float64(T)
    return softmax_gather_grad(x, idx, g, T), g


def entropy_from_logits_bwd(x, dentropy, T):
    """Gradient of sum_r u_r * H_r with respect to the logits (fp64), u = dentropy.

    H = -sum_j p_j log p_j with p = softmax(x / T) (the entropy of [axolotl],
    "1. benchmarks/bench_entropy.py"); dH/dx_k = -(p_k / T) (log p_k + H).  The pages
    print no entropy backward: this is the derivative of their definition.  Rows with
    u_r == 0 are +0.0 (as for the other backward passes).  Returns (dlogits, g) with
    g_r = -u_r / T.
    """
    z, lse = log_softmax_rows(x, T)
    H = entropy_from_logits(x, T)
    g = -np.asarray(dentropy, dtype=np.float64) / np.float64(T)
    with np.errstate(invalid="ignore", over="ignore"):
        logp = z - lse[:, None]
        p = np.exp(logp)
        d = g[:, None] * np.where(p == 0.0, 0.0, p * (logp + H[:, None]))
    d[g == 0.0] = 0.0                         # +0.0 rows, also for u == -0.0
    return d, g


def grpo_seq_terms(logp, old_logp, ref_logp, adv_seq, mask, dloss, B, L, beta, eps_low, eps_high):
    """Sequence-level GRPO terms (fp64) for B sequences of L tokens.

    [Liger-bwd], "Code analysis", shows a sequence-level backward kernel
    (``_grpo_loss_bwd_kernel_seq``) whose token KL gradient beta * (1 - exp(ref - logp))
    is weighted by that token's dloss inside the kernel while the policy-gradient part
    arrives already computed per sequence; the pages print no ratio.  Reading taken
    here: the importance ratio of sequence b is the length-normalised sequence ratio

        s_b  = exp( sum_t m_bt (logp_bt - old_bt) / n_b ),   n_b = sum_t m_bt
        pg_b = -min(s_b A_b, clip(s_b, 1 - eps_low, 1 + eps_high) A_b)

    every unmasked token carries loss_t = pg_b + kl_t (kl_t the token k3 term), and the
    objective is J = sum_t dloss_t loss_t.  Hence, for an unmasked token t of b,

        dJ/dlogp_t = W_b dpg_b/dlogp_t + beta (1 - exp(ref_t - logp_t)) dloss_t,
        W_b = sum_t dloss_bt,  dpg_b/dlogp_t = -A_b s_b / n_b (unclipped branch, ties
        included) or 0 (clipping binds);

    masked tokens have loss = kl = dlogp = +0.0; a sequence without tokens has s_b = 1.
    """
    logp = np.asarray(logp, dtype=np.float64).reshape(B, L)
    m = np.ones((B, L), dtype=bool) if mask is None else (np.asarray(mask).reshape(B, L) != 0)
    dl = np.asarray(dloss, dtype=np.float64).reshape(B, L)
    A = np.asarray(adv_seq, dtype=np.float64)
    old = logp if old_logp is None else np.asarray(old_logp, dtype=np.float64).reshape(B, L)
    n = m.sum(axis=1)
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        log_s = np.where(n > 0, np.where(m, logp - old, 0.0).sum(axis=1) / np.maximum(n, 1), 0.0)
        s = np.exp(log_s)
        clipped = np.clip(s, 1.0 - eps_low, 1.0 + eps_high)
        pg = -np.minimum(s * A, clipped * A)
        is_clipped = (clipped * A) < (s * A)
        dpg = np.where((s * A) <= (clipped * A), -A * s / np.maximum(n, 1), 0.0)
        W = np.where(m, dl, 0.0).sum(axis=1)
        if beta != 0.0:
            d = np.asarray(ref_logp, dtype=np.float64).reshape(B, L) - logp
            kl = beta * (np.expm1(d) - d)
            dkl = beta * (1.0 - np.exp(d))
        else:
            kl = np.zeros((B, L))
            dkl = np.zeros((B, L))
        loss = pg[:, None] + kl
        dlogp = (W * dpg)[:, None] + dkl * dl
    z = np.zeros((B, L))
    return {
        "seq_ratio": s, "seq_pg": pg, "seq_is_clipped": is_clipped,
        "loss": np.where(m, loss, z).reshape(-1), "kl": np.where(m, kl, z).reshape(-1),
        "dlogp": np.where(m, dlogp, z).reshape(-1),
    }


def grpo_seq_loss_bwd(x, idx, old_logp, ref_logp, adv_seq, mask, dloss, B, L, T, beta, eps_low, eps_high):
    """dlogits of the sequence-level objective (fp64): the per-token dlogp of
    grpo_seq_terms spread over each row as (dlogp / T) (1[j == idx] - p_j), with the
    zero-row rule of softmax_gather_grad.  Returns (dlogits, g, terms)."""
    logp, _ = selective_log_softmax(x, idx, T)
    terms = grpo_seq_terms(logp, old_logp, ref_logp, adv_seq, mask, dloss, B, L, beta, eps_low, eps_high)
    g = terms["dlogp"] / np.float64(T)
    return softmax_gather_grad(x, idx, g, T), g, terms


def fused_linear_grpo(h, W, idx, old_logp, ref_logp, adv_row, mask, dloss, T, beta, eps_low, eps_high):
    """The GRPO loss on top of the LM head, with the gradients of the hidden states and
    of the head weight (fp64).

    [Liger-TRL], section 3: the logits are the LM head applied to the hidden states of
    the rows, x = h W^T ([R, H] x [H, V]); section 4: the loss of each chunk of rows
    computes, during its forward, the gradient of its input chunk and of the head
    weight, and the weight gradient is accumulated over the chunks.  Splitting the rows
    into chunks changes no value, so the definition is written on all rows at once:

        x = h W^T,  loss / logp / ... = grpo_loss_fwd(x),  dx = grpo_loss_bwd(x)[0],
        grad_h = dx W,  grad_W = dx^T h        (J = sum_r dloss_r loss_r)

    Returns (fwd dict as grpo_loss_fwd, grad_h [R, H], grad_W [V, H], dx [R, V]).
    """
    h = np.asarray(h, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    x = h @ W.T
    fwd = grpo_loss_fwd(x, idx, old_logp, ref_logp, adv_row, mask, T, beta, eps_low, eps_high)
    dx, _ = grpo_loss_bwd(x, idx, old_logp, ref_logp, adv_row, mask, dloss, T, beta, eps_low, eps_high)
    grad_h = dx @ W
    grad_W = dx.T @ h
    return fwd, grad_h, grad_W, dx
