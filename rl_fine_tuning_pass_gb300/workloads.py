"""Seeded synthetic inputs for the row pass (shared by the tests, the benchmark
and the oracle checks).

This module draws random numbers and builds masks; it holds none of the row
pass's arithmetic (no softmax, no log-probabilities, no loss).  Quantities the
row pass needs but that depend on its own results, such as an ``old_logp`` that
sits close to the current ``logp``, are returned as *offsets* (``old_offset``,
``ref_offset``); the caller adds them to a logp it computed itself.

Workloads (the shapes and distributions of the pages' benchmarks):

* ``tiny_fp32``            B=2,  L=16,   V=512,    fp32 -- the small case the oracle
                           finishes in well under a second.
* ``grpo_b4_l512_v32000``  B=4,  L=512,  V=32000,  bf16 -- the GRPO backward workload
                           of the Liger-Kernel GRPO Loss Backward write-up
                           ("Why it's good": (B, L, V, zero-grad%) = (4, 512, 32000, 50%)).
* ``entropy_slsm_b16_l4096_v32000``  B=16, L=4096, V=32000, bf16 -- the entropy and
                           selective-log-softmax benchmark size of the axolotl write-up
                           ("Why it's good", "1. Performance": B=16, L=4096), with a
                           non-contiguous variant (``logits[:, :-1, :]`` of a
                           [16, 4097, V] tensor, as in its ``benchmark_noncontiguous``).
* ``grpo_qwen3_b16_l1024_v151936``  B=16 (4 prompts x 4 completions), L=1024,
                           V=151936 (a Qwen3-0.6B-shaped LM head, no weights).
* ``sweep_b16_l4096_v151936``       B=16, L=4096, V=151936 (~20 GB bf16 logits),
                           T=0.7; beta (0.04 by default, or 0) and the zero-advantage
                           fraction (8 of 16 sequences by default) swept.
* ``linear_qwen3_b16_l1024_h1024_v151936``  the Qwen3-shaped GRPO batch above given as
                           hidden states [B*L, H=1024] and an LM-head weight [V, H]
                           (Qwen3-0.6B's hidden size), bf16, for the loss on top of the
                           head (``generate_linear``).  h ~ N(0, 1), W ~ N(0, w_sigma^2)
                           with w_sigma = sigma / sqrt(H), so the logits have the same
                           N(0, sigma^2) spread as the logits workloads.

The public GRPO runs the pages cite use datasets (gsm8k, TLDR) and trained
weights that are not available here; these synthetic tensors stand in for the
LM-head logits such runs produce, with the same shapes.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

__all__ = ["WorkloadSpec", "WORKLOADS", "get", "Inputs", "generate", "logits_rows", "LinearInputs",
           "generate_linear", "sample_rows"]


@dataclasses.dataclass(frozen=True)
class WorkloadSpec:
    name: str
    B: int
    L: int
    V: int
    dtype: str                 # "bf16" or "fp32"
    sigma: float               # logits ~ N(0, sigma^2)
    T: float
    beta: float
    eps_low: float
    eps_high: float
    adv: str                   # how advantages are drawn (see _advantages)
    mask: str                  # "none" | "trailing10" | "uniform_len"
    old_sigma: Optional[float]  # old_logp = logp + N(0, old_sigma^2); None => no old_logp
    ref_sigma: Optional[float]  # ref_logp = logp + N(0, ref_sigma^2); None => no ref_logp
    peaked_frac: float = 0.0   # fraction of rows with one logit raised by peak_height
    peak_height: float = 20.0
    group_size: int = 1        # completions per prompt (for group-normalised advantages)
    zero_adv_seqs: int = 0     # for adv == "sweep": number of sequences with A == 0
    strided: bool = False      # logits as logits[:, :-1, :] of a [B, L+1, V] tensor
    H: int = 0                 # hidden size of the LM-head workloads (logits = h W^T)

    @property
    def rows(self) -> int:
        return self.B * self.L

    @property
    def elem_size(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def with_(self, **kw) -> "WorkloadSpec":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny_fp32": WorkloadSpec(
        "tiny_fp32", B=2, L=16, V=512, dtype="fp32", sigma=2.0, T=1.0, beta=0.04,
        eps_low=0.2, eps_high=0.2, adv="plus_minus_one", mask="none",
        old_sigma=0.1, ref_sigma=0.05),
    "grpo_b4_l512_v32000": WorkloadSpec(
        "grpo_b4_l512_v32000", B=4, L=512, V=32000, dtype="bf16", sigma=2.0, T=0.9, beta=0.0,
        eps_low=0.2, eps_high=0.2, adv="half_zero", mask="trailing10",
        old_sigma=0.15, ref_sigma=None),
    "entropy_slsm_b16_l4096_v32000": WorkloadSpec(
        "entropy_slsm_b16_l4096_v32000", B=16, L=4096, V=32000, dtype="bf16", sigma=3.0, T=1.0,
        beta=0.0, eps_low=0.2, eps_high=0.2, adv="none", mask="none",
        old_sigma=None, ref_sigma=None, peaked_frac=0.05, peak_height=20.0),
    "grpo_qwen3_b16_l1024_v151936": WorkloadSpec(
        "grpo_qwen3_b16_l1024_v151936", B=16, L=1024, V=151936, dtype="bf16", sigma=2.0, T=1.0,
        beta=0.04, eps_low=0.2, eps_high=0.28, adv="group_bernoulli", mask="uniform_len",
        old_sigma=0.15, ref_sigma=0.05, group_size=4),
    "linear_qwen3_b16_l1024_h1024_v151936": WorkloadSpec(
        "linear_qwen3_b16_l1024_h1024_v151936", B=16, L=1024, V=151936, dtype="bf16", sigma=2.0, T=1.0,
        beta=0.04, eps_low=0.2, eps_high=0.28, adv="group_bernoulli", mask="uniform_len",
        old_sigma=0.15, ref_sigma=0.05, group_size=4, H=1024),
    "sweep_b16_l4096_v151936": WorkloadSpec(
        "sweep_b16_l4096_v151936", B=16, L=4096, V=151936, dtype="bf16", sigma=2.0, T=0.7,
        beta=0.04, eps_low=0.2, eps_high=0.2, adv="sweep", mask="none",
        old_sigma=0.05, ref_sigma=0.05, zero_adv_seqs=8),
}


def get(name: str, **overrides) -> WorkloadSpec:
    spec = WORKLOADS[name]
    return spec.with_(**overrides) if overrides else spec


# Independent streams per component so that changing how one tensor is drawn
# never shifts another.
_STREAM = {"logits": 1, "idx": 2, "old": 3, "ref": 4, "adv": 5, "mask": 6, "peak": 7, "hidden": 8, "head": 9}


def _gen(seed: int, what: str, device="cpu", chunk: int = 0) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + _STREAM[what] * 7919 + chunk * 104_729) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


@dataclasses.dataclass
class Inputs:
    spec: WorkloadSpec
    logits: Optional[torch.Tensor]     # [B, L, V] (possibly a strided view), bf16 or fp32; None if not drawn
    idx: torch.Tensor                  # [B*L] int64
    adv: torch.Tensor                  # [B] fp32
    mask: Optional[torch.Tensor]       # [B*L] uint8, or None (all tokens count)
    dloss: torch.Tensor                # [B*L] fp32: mask / (B * completion length)
    old_offset: Optional[torch.Tensor]  # [B*L] fp32 noise to add to logp, or None
    ref_offset: Optional[torch.Tensor]  # [B*L] fp32 noise to add to logp, or None
    upstream: torch.Tensor             # [B*L] fp32 upstream grad for the selective-log-softmax bwd
    lengths: torch.Tensor              # [B] int64 completion lengths

    @property
    def rows(self) -> int:
        return self.spec.rows


def _torch_dtype(d: str):
    return torch.bfloat16 if d == "bf16" else torch.float32


def _fill_logits(spec: WorkloadSpec, seed: int, device, rows_per_chunk: int) -> torch.Tensor:
    """Logits ~ N(0, sigma^2), drawn in fp32 in row chunks (bounded temporary memory)
    and rounded to the storage dtype.  Each chunk has its own seeded generator, so for
    a given device type and ``rows_per_chunk`` the values are reproducible."""
    B, L, V = spec.B, spec.L, spec.V
    Lp = L + 1 if spec.strided else L
    base = torch.empty((B * Lp, V), dtype=_torch_dtype(spec.dtype), device=device)
    dev_type = torch.device(device).type
    for c, r0 in enumerate(range(0, B * Lp, rows_per_chunk)):
        r1 = min(B * Lp, r0 + rows_per_chunk)
        g = _gen(seed, "logits", dev_type, chunk=c)
        blk = torch.randn((r1 - r0, V), generator=g, device=device, dtype=torch.float32)
        blk.mul_(spec.sigma)
        base[r0:r1].copy_(blk)
        del blk
    base = base.view(B, Lp, V)
    return base[:, :L, :] if spec.strided else base


def _advantages(spec: WorkloadSpec, seed: int) -> torch.Tensor:
    """Per-sequence advantages A[b] (fp32, on the host).

    * plus_minus_one:  A = [+1, -1, +1, ...]
    * half_zero:       A = [N(0,1), 0, N(0,1), 0, ...] (every second sequence exactly 0)
    * group_bernoulli: rewards ~ Bernoulli(0.5) per completion, normalised within each
                       group of ``group_size`` completions of one prompt:
                       (R - mean) / (std + 1e-4), population std.  A group whose rewards
                       are all equal gets A == 0 exactly (R - mean is exactly 0).
                       This is the group-relative advantage of GRPO with a verifiable
                       (0/1) reward (Liger GRPO meets TRL, "2. The core principle that
                       sets GRPO apart from PPO"); the row pass only consumes A.
    * sweep:           the first ``zero_adv_seqs`` sequences (in a seeded order) get
                       A == 0, the others A ~ N(0,1).
    * none:            zeros (workloads that do not run the GRPO loss).
    """
    B = spec.B
    g = _gen(seed, "adv")
    if spec.adv == "plus_minus_one":
        return torch.tensor([1.0 if b % 2 == 0 else -1.0 for b in range(B)], dtype=torch.float32)
    if spec.adv == "half_zero":
        a = torch.randn(B, generator=g, dtype=torch.float64)
        a[1::2] = 0.0
        return a.float()
    if spec.adv == "group_bernoulli":
        G = spec.group_size
        assert B % G == 0
        r = torch.bernoulli(torch.full((B,), 0.5, dtype=torch.float64), generator=g)
        r = r.view(B // G, G)
        mean = r.mean(dim=1, keepdim=True)
        std = r.std(dim=1, unbiased=False, keepdim=True)
        return ((r - mean) / (std + 1e-4)).reshape(B).float()
    if spec.adv == "sweep":
        a = torch.randn(B, generator=g, dtype=torch.float64)
        order = torch.randperm(B, generator=g)
        a[order[: spec.zero_adv_seqs]] = 0.0
        return a.float()
    if spec.adv == "none":
        return torch.zeros(B, dtype=torch.float32)
    raise ValueError(spec.adv)


def _lengths(spec: WorkloadSpec, seed: int) -> torch.Tensor:
    B, L = spec.B, spec.L
    if spec.mask == "none":
        return torch.full((B,), L, dtype=torch.int64)
    if spec.mask == "trailing10":
        return torch.full((B,), L - (L // 10), dtype=torch.int64)   # 10% trailing padding
    if spec.mask == "uniform_len":
        g = _gen(seed, "mask")
        lo = L // 4
        return torch.randint(lo, L + 1, (B,), generator=g, dtype=torch.int64)
    raise ValueError(spec.mask)


def _row_inputs(spec: WorkloadSpec, seed: int):
    """Advantages, mask, per-token loss weights, old/ref offsets, upstream gradient and
    completion lengths (host tensors)."""
    B, L, R = spec.B, spec.L, spec.rows
    adv = _advantages(spec, seed)
    lengths = _lengths(spec, seed)
    pos = torch.arange(L, dtype=torch.int64)[None, :]
    mask_bl = (pos < lengths[:, None]).to(torch.uint8)
    mask = None if spec.mask == "none" else mask_bl.reshape(R)
    # per-token loss weight: mean over each completion, then mean over the batch
    dloss = (mask_bl.double() / (B * lengths[:, None].double())).float().reshape(R)
    old_offset = ref_offset = None
    if spec.old_sigma is not None:
        old_offset = (torch.randn(R, generator=_gen(seed, "old"), dtype=torch.float64) * spec.old_sigma).float()
    if spec.ref_sigma is not None:
        ref_offset = (torch.randn(R, generator=_gen(seed, "ref"), dtype=torch.float64) * spec.ref_sigma).float()
    upstream = torch.full((R,), 1.0 / R, dtype=torch.float32)
    return adv, mask, dloss, old_offset, ref_offset, upstream, lengths


def _idx(spec: WorkloadSpec, seed: int) -> torch.Tensor:
    return torch.randint(0, spec.V, (spec.rows,), generator=_gen(seed, "idx"), dtype=torch.int64)


def _peaks(spec: WorkloadSpec, seed: int, idx: torch.Tensor):
    """Rows (sorted) and columns of the peaked logits: a seeded choice of
    round(peaked_frac * R) rows; even-numbered peaked rows are peaked on the sampled token,
    odd ones on a random column."""
    R, V = spec.rows, spec.V
    gp = _gen(seed, "peak")
    n_peak = int(round(spec.peaked_frac * R))
    rows = torch.sort(torch.randperm(R, generator=gp)[:n_peak]).values
    cols_rand = torch.randint(0, V, (n_peak,), generator=gp, dtype=torch.int64)
    cols = torch.where(torch.arange(n_peak) % 2 == 0, idx.cpu()[rows], cols_rand)
    return rows, cols


def logits_rows(spec: WorkloadSpec, seed: int, r0: int, r1: int, device="cpu",
                rows_per_chunk: int = 4096) -> torch.Tensor:
    """Rows [r0, r1) of the [B*L, V] logits, with the values ``generate`` gives them on the
    same device type, drawing only the generator chunks that hold them (a bounded sample of
    a batch too large to draw whole on the host)."""
    B, L, V = spec.B, spec.L, spec.V
    Lp = L + 1 if spec.strided else L
    dev_type = torch.device(device).type
    flat = torch.arange(r0, r1, dtype=torch.int64)
    base_rows = (flat // L) * Lp + flat % L  # rows of the [B*Lp, V] buffer
    out = torch.empty((r1 - r0, V), dtype=_torch_dtype(spec.dtype), device=device)
    lo, hi = int(base_rows[0]) if len(flat) else 0, int(base_rows[-1]) + 1 if len(flat) else 0
    for c in range(lo // rows_per_chunk, (hi + rows_per_chunk - 1) // rows_per_chunk):
        c0, c1 = c * rows_per_chunk, min(B * Lp, (c + 1) * rows_per_chunk)
        g = _gen(seed, "logits", dev_type, chunk=c)
        blk = torch.randn((c1 - c0, V), generator=g, device=device, dtype=torch.float32)
        blk.mul_(spec.sigma)
        sel = (base_rows >= c0) & (base_rows < c1)
        if bool(sel.any()):
            out[sel.to(out.device)] = blk[(base_rows[sel] - c0).to(blk.device)].to(out.dtype)
        del blk
    if spec.peaked_frac > 0.0:
        rows, cols = _peaks(spec, seed, _idx(spec, seed))
        keep = (rows >= r0) & (rows < r1)
        rr, cc = (rows[keep] - r0).to(out.device), cols[keep].to(out.device)
        out[rr, cc] = (out[rr, cc].float() + spec.peak_height).to(out.dtype)
    return out


def generate(spec: WorkloadSpec, seed: int = 0, device="cpu", rows_per_chunk: int = 4096,
             with_logits: bool = True) -> Inputs:
    """All inputs of one workload, seeded.  Large logits should be generated with
    ``device='cuda'`` (drawn on the GPU in row chunks); the small per-row arrays are
    always drawn on the host and then moved to ``device``.  ``with_logits=False`` leaves
    the logits out (``logits`` is None; ``logits_rows`` draws a slice of them)."""
    B, L, V, R = spec.B, spec.L, spec.V, spec.rows
    logits = _fill_logits(spec, seed, device, rows_per_chunk) if with_logits else None

    idx = _idx(spec, seed)

    if spec.peaked_frac > 0.0 and with_logits:
        rows, cols = _peaks(spec, seed, idx)
        flat = logits.reshape(R, V) if not spec.strided else None
        for k in range(0, len(rows), 65536):
            rr, cc = rows[k:k + 65536], cols[k:k + 65536]
            if flat is not None:
                rd, cd = rr.to(logits.device), cc.to(logits.device)
                vals = flat[rd, cd].float() + spec.peak_height
                flat[rd, cd] = vals.to(flat.dtype)
            else:
                b, l = (rr // L).to(logits.device), (rr % L).to(logits.device)
                cd = cc.to(logits.device)
                vals = logits[b, l, cd].float() + spec.peak_height
                logits[b, l, cd] = vals.to(logits.dtype)

    adv, mask, dloss, old_offset, ref_offset, upstream, lengths = _row_inputs(spec, seed)
    mv = lambda t: None if t is None else t.to(device)
    return Inputs(spec, logits, mv(idx), mv(adv), mv(mask), mv(dloss), mv(old_offset), mv(ref_offset),
                  mv(upstream), lengths)


def sample_rows(R: int, k: int, seed: int = 0) -> np.ndarray:
    """k distinct row indices in [0, R), sorted, always including the first and the
    last row, for checking large workloads row by row against the oracle."""
    if k >= R:
        return np.arange(R, dtype=np.int64)
    rng = np.random.default_rng(seed + 12345)
    inner = rng.choice(np.arange(1, R - 1), size=max(k - 2, 0), replace=False)
    return np.unique(np.concatenate([[0, R - 1], inner]).astype(np.int64))


@dataclasses.dataclass
class LinearInputs:
    spec: WorkloadSpec
    hidden: torch.Tensor               # [B*L, H] bf16 hidden states entering the LM head
    weight: torch.Tensor               # [V, H] bf16 LM-head weight
    idx: torch.Tensor                  # [B*L] int64
    adv: torch.Tensor                  # [B] fp32
    mask: Optional[torch.Tensor]       # [B*L] uint8 or None
    dloss: torch.Tensor                # [B*L] fp32
    old_offset: Optional[torch.Tensor]
    ref_offset: Optional[torch.Tensor]
    lengths: torch.Tensor


def generate_linear(spec: WorkloadSpec, seed: int = 0, device="cpu") -> LinearInputs:
    """Inputs of the GRPO loss on top of the LM head: hidden states h ~ N(0, 1) and a head
    weight W ~ N(0, (sigma / sqrt(H))^2), both bf16, drawn in fp32 with their own seeded
    streams; the per-row inputs as in ``generate``."""
    B, L, V, H, R = spec.B, spec.L, spec.V, spec.H, spec.rows
    assert H > 0, "not an LM-head workload"
    dev_type = torch.device(device).type
    h = torch.randn((R, H), generator=_gen(seed, "hidden", dev_type), device=device, dtype=torch.float32)
    W = torch.randn((V, H), generator=_gen(seed, "head", dev_type), device=device, dtype=torch.float32)
    W.mul_(spec.sigma / float(np.sqrt(H)))
    idx = torch.randint(0, V, (R,), generator=_gen(seed, "idx"), dtype=torch.int64)
    adv, mask, dloss, old_offset, ref_offset, _, lengths = _row_inputs(spec, seed)
    mv = lambda t: None if t is None else t.to(device)
    return LinearInputs(spec, h.to(torch.bfloat16), W.to(torch.bfloat16), mv(idx), mv(adv), mv(mask), mv(dloss),
                        mv(old_offset), mv(ref_offset), lengths)
