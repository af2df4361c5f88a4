"""The GRPO loss on top of the LM head (grpo_fused_linear) against the oracle's
fused_linear_grpo: forward outputs on every row, and the hidden-state and head-weight
gradients element by element (GPU).

Tolerances: the forward outputs as in parity_util (the logits are formed in fp32 by the
GEMM, a relative error of ~1e-7 of |h||w|).  The gradients take dlogits rounded to bf16
(relative 2^-9 per element) into the backward GEMMs, so an element of grad_h may move by
2^-9 sum_j |dx_rj| |W_jk| and one of grad_W by 2^-9 sum_r |dx_rj| |h_rk|; the tests allow
twice that, plus 1e-5 relative and fp32 accumulation.
"""

import numpy as np
import pytest
import torch

import oracle
from parity_util import ambiguous_rows, assert_scalar_close, rows_f64
from rl_fine_tuning_pass_gb300 import binding as rp
from rl_fine_tuning_pass_gb300 import workloads as W

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _library():
    from rl_fine_tuning_pass_gb300.build import build
    build()
    rp.load_library()


def problem(B, L, H, V, seed, beta, masked=True, zero_adv=True):
    g = torch.Generator().manual_seed(seed)
    R = B * L
    h = torch.randn(R, H, generator=g).to(torch.bfloat16)
    Wt = (torch.randn(V, H, generator=g) * (2.0 / np.sqrt(H))).to(torch.bfloat16)
    idx = torch.randint(0, V, (R,), generator=g)
    adv = torch.randn(B, generator=g).float()
    if zero_adv:
        adv[0] = 0.0
    mask = (torch.rand(R, generator=g) > 0.2).to(torch.uint8) if masked else None
    dloss = (torch.rand(R, generator=g) + 0.1).float()
    if mask is not None:
        dloss *= mask.float()
    T = 0.9
    hf, Wf = rows_f64(h), rows_f64(Wt)
    lp0, _ = oracle.selective_log_softmax(hf @ Wf.T, idx.numpy(), T)
    old = oracle.round_to_fp32(lp0 + torch.randn(R, generator=g).double().numpy() * 0.2)
    ref = oracle.round_to_fp32(lp0 + torch.randn(R, generator=g).double().numpy() * 0.1) if beta else None
    return dict(h=h, W=Wt, idx=idx, adv=adv, mask=mask, dloss=dloss, old=old, ref=ref, T=T, beta=beta, el=0.2,
                eh=0.28, B=B, L=L, hf=hf, Wf=Wf)


def run_gpu(pb, chunk, grad_weight=None):
    t = lambda a, dt=torch.float32: None if a is None else torch.as_tensor(a, dtype=dt).to(DEV)
    dev_err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = rp.grpo_fused_linear(pb["h"].to(DEV), pb["W"].to(DEV), t(pb["idx"], torch.int64), t(pb["adv"]),
                               t(pb["dloss"]), B=pb["B"], L=pb["L"], T=pb["T"], beta=pb["beta"], eps_low=pb["el"],
                               eps_high=pb["eh"], old_logp=t(pb["old"]), ref_logp=t(pb["ref"]),
                               mask=t(pb["mask"], torch.uint8), chunk_rows=chunk, grad_weight=grad_weight,
                               dev_err=dev_err)
    torch.cuda.synchronize()
    return out, int(dev_err.item())


def check_against_oracle(pb, out, what, grad_weight_scale=1.0):
    R = pb["B"] * pb["L"]
    adv_row = oracle.per_row(pb["adv"].numpy(), pb["L"])
    mask = None if pb["mask"] is None else pb["mask"].numpy()
    f, gh, gW, dx = oracle.fused_linear_grpo(pb["hf"], pb["Wf"], pb["idx"].numpy(), pb["old"], pb["ref"], adv_row,
                                             mask, pb["dloss"].double().numpy(), pb["T"], pb["beta"], pb["el"],
                                             pb["eh"])
    for k in ("loss", "logp", "lse", "kl", "entropy"):
        assert_scalar_close(out[k], f[k], f"{what} {k}")
    amb = ambiguous_rows(f["ratio"], adv_row, mask, pb["el"], pb["eh"])
    clip = out["is_clipped"].cpu().numpy().astype(bool)
    assert np.array_equal(clip[~amb], f["is_clipped"][~amb]), f"{what} is_clipped"
    assert amb.sum() == 0, f"{what}: a row sits on a clip boundary; pick another seed"

    got_h = out["grad_hidden"].double().cpu().numpy()
    bound_h = 2.0 ** -8 * (np.abs(dx) @ np.abs(pb["Wf"])) + 1e-5 * np.abs(gh) + 1e-7
    bad = np.abs(got_h - gh) > bound_h
    assert not bad.any(), f"{what} grad_hidden: {bad.sum()} elements out, worst {np.abs(got_h - gh)[bad].max():.3g}"
    zero_rows = np.all(dx == 0.0, axis=1)
    assert np.all(got_h[zero_rows] == 0.0), f"{what}: rows with a zero gradient must get grad_hidden 0"

    got_W = out["grad_weight"].double().cpu().numpy()
    bound_W = grad_weight_scale * (2.0 ** -8 * (np.abs(dx).T @ np.abs(pb["hf"])) + 1e-5 * np.abs(gW)) + 1e-7
    bad = np.abs(got_W - grad_weight_scale * gW) > bound_W
    assert not bad.any(), f"{what} grad_weight: {bad.sum()} elements out"
    return f, gh, gW


@pytest.mark.parametrize("V,chunk,beta", [(1000, 16, 0.04), (1003, 16, 0.0), (517, 64, 0.04), (2048, 7, 0.0)])
def test_fused_linear_every_row(V, chunk, beta):
    """Ragged last chunk (42 rows in chunks of 16 / 7), V with and without a multiple of 8,
    masked rows, a zero-advantage sequence, beta on and off."""
    pb = problem(2, 21, 64, V, seed=V + chunk, beta=beta)
    out, err = run_gpu(pb, chunk)
    assert err == 0
    check_against_oracle(pb, out, f"fused linear V={V} chunk={chunk}")


def test_fused_linear_without_a_mask():
    """mask = NULL: every row counts, the chunks are the batch's rows in order."""
    pb = problem(2, 21, 64, 1000, seed=11, beta=0.04, masked=False)
    out, err = run_gpu(pb, 16)
    assert err == 0
    check_against_oracle(pb, out, "fused linear without a mask")


@pytest.mark.parametrize("chunk", [5, 16, 64, 200])
def test_fused_linear_packs_unmasked_rows_across_padding(chunk):
    """Completions of different lengths with trailing padding (60 % of the rows masked, one
    sequence fully masked): the chunks take only unmasked rows, so they cross sequence
    boundaries, and the chunks after the last unmasked row find nothing to do.  Masked
    rows get zero outputs and an exactly zero grad_hidden row."""
    B, L, H, V = 4, 50, 64, 1003
    pb = problem(B, L, H, V, seed=100 + chunk, beta=0.04)
    lengths = [37, 0, 12, 31]
    mask = torch.zeros(B * L, dtype=torch.uint8)
    for b, n in enumerate(lengths):
        mask[b * L:b * L + n] = 1
    pb["mask"] = mask
    pb["dloss"] = (pb["dloss"] + 0.1) * mask.float()
    out, err = run_gpu(pb, chunk)
    assert err == 0
    check_against_oracle(pb, out, f"packed rows, chunk {chunk}")
    m = mask.to(DEV).bool()
    for k in ("loss", "logp", "lse", "kl", "entropy"):
        assert torch.all(out[k][~m] == 0), k
    assert torch.all(out["grad_hidden"][~m] == 0)


def test_fused_linear_every_row_masked():
    """No unmasked row: every output and grad_hidden row is zero and grad_weight keeps its
    values bit for bit (no chunk holds a row, so no GEMM adds anything)."""
    pb = problem(2, 21, 64, 517, seed=9, beta=0.04)
    pb["mask"] = torch.zeros(42, dtype=torch.uint8)
    pb["dloss"] = torch.zeros(42)
    gW = torch.randn(517, 64, generator=torch.Generator().manual_seed(1)).to(DEV)
    before = gW.clone()
    out, err = run_gpu(pb, 16, grad_weight=gW)
    assert err == 0
    for k in ("loss", "logp", "lse", "kl", "entropy", "grad_hidden"):
        assert torch.all(out[k] == 0), k
    assert torch.all(out["is_clipped"] == 0)
    assert torch.equal(gW, before)


def test_fused_linear_accumulates_weight_gradient_and_chunking_is_invisible():
    """grad_weight is accumulated into the given tensor; the chunk size changes the row
    pass's outputs not at all, the GEMMs' outputs only by their fp32 summation order."""
    pb = problem(2, 24, 128, 3000, seed=5, beta=0.04)
    gW = torch.zeros(3000, 128, dtype=torch.float32, device=DEV)
    out1, _ = run_gpu(pb, 1000, grad_weight=gW)
    out2, _ = run_gpu(pb, 5, grad_weight=gW)      # second call adds to the first
    check_against_oracle(pb, out2, "two accumulated calls", grad_weight_scale=2.0)
    for k in ("loss", "logp", "lse", "entropy"):
        assert torch.equal(out1[k], out2[k]), k   # the row pass does not depend on the chunking
    # grad_hidden comes from a GEMM whose summation order depends on the chunk's width
    assert torch.allclose(out1["grad_hidden"], out2["grad_hidden"], rtol=1e-4, atol=1e-7)


def test_fused_linear_qwen3_head_rows():
    """H = 1024 (Qwen3-0.6B's hidden size), V = 32000, 512 rows in chunks of 128: every
    row against the oracle."""
    spec = W.get("linear_qwen3_b16_l1024_h1024_v151936", B=4, L=128, V=32000)
    li = W.generate_linear(spec, 0, device="cpu")
    T = spec.T
    hf, Wf = rows_f64(li.hidden), rows_f64(li.weight)
    lp0, _ = oracle.selective_log_softmax(hf @ Wf.T, li.idx.numpy(), T)
    old = oracle.round_to_fp32(lp0 + li.old_offset.double().numpy())
    ref = oracle.round_to_fp32(lp0 + li.ref_offset.double().numpy())
    pb = dict(h=li.hidden, W=li.weight, idx=li.idx, adv=li.adv, mask=li.mask, dloss=li.dloss, old=old, ref=ref, T=T,
              beta=spec.beta, el=spec.eps_low, eh=spec.eps_high, B=spec.B, L=spec.L, hf=hf, Wf=Wf)
    out, err = run_gpu(pb, 128)
    assert err == 0
    check_against_oracle(pb, out, "qwen3 head")


def test_fused_linear_bench_shape_against_oracle():
    """The benchmark's LM-head shape (H = 1024, V = 151936: fp32 logit rows of 594 KB, the
    last 256-column tile half empty) in its launch configuration (chunks of 2048 rows),
    with one full chunk and a ragged second one (2148 rows): the forward outputs of every
    row, grad_hidden on sampled rows and grad_weight on sampled vocabulary rows against the
    oracle on all rows."""
    spec = W.get("linear_qwen3_b16_l1024_h1024_v151936", B=4, L=537)
    li = W.generate_linear(spec, 0, device="cpu")
    R, V, H, T = spec.rows, spec.V, spec.H, spec.T
    hf, Wf = rows_f64(li.hidden), rows_f64(li.weight)
    lp0, _ = oracle.selective_log_softmax(hf @ Wf.T, li.idx.numpy(), T)
    old = oracle.round_to_fp32(lp0 + li.old_offset.double().numpy())
    ref = oracle.round_to_fp32(lp0 + li.ref_offset.double().numpy())
    pb = dict(h=li.hidden, W=li.weight, idx=li.idx, adv=li.adv, mask=li.mask, dloss=li.dloss, old=old, ref=ref, T=T,
              beta=spec.beta, el=spec.eps_low, eh=spec.eps_high, B=spec.B, L=spec.L, hf=hf, Wf=Wf)
    out, err = run_gpu(pb, 2048)
    assert err == 0
    adv_row = oracle.per_row(li.adv.numpy(), spec.L)
    mask = li.mask.numpy()
    f, gh, gW, dx = oracle.fused_linear_grpo(hf, Wf, li.idx.numpy(), old, ref, adv_row, mask,
                                             li.dloss.double().numpy(), T, spec.beta, spec.eps_low, spec.eps_high)
    for k in ("loss", "logp", "lse", "kl", "entropy"):
        assert_scalar_close(out[k], f[k], f"bench shape {k}")
    amb = ambiguous_rows(f["ratio"], adv_row, mask, spec.eps_low, spec.eps_high)
    clip = out["is_clipped"].cpu().numpy().astype(bool)
    assert np.array_equal(clip[~amb], f["is_clipped"][~amb]), "bench shape is_clipped"
    assert (mask == 0).any() and (mask != 0).any()

    rows = np.unique(np.concatenate([W.sample_rows(R, 48, 1), [0, 2047, 2048, R - 1]]))
    got_h = out["grad_hidden"].double().cpu().numpy()[rows]
    bound_h = 2.0 ** -8 * (np.abs(dx[rows]) @ np.abs(Wf)) + 1e-5 * np.abs(gh[rows]) + 1e-7
    bad = np.abs(got_h - gh[rows]) > bound_h
    assert not bad.any(), f"grad_hidden: {bad.sum()} elements out, worst {np.abs(got_h - gh[rows])[bad].max():.3g}"
    assert np.all(got_h[np.all(dx[rows] == 0.0, axis=1)] == 0.0)

    cols = np.unique(np.concatenate([W.sample_rows(V, 40, 2), li.idx.numpy()[rows[:8]],
                                     np.arange(V - 130, V), [V - 257, 255, 256]]))
    got_W = out["grad_weight"].double().cpu().numpy()[cols]
    bound_W = 2.0 ** -8 * (np.abs(dx[:, cols]).T @ np.abs(hf)) + 1e-5 * np.abs(gW[cols]) + 1e-7
    bad = np.abs(got_W - gW[cols]) > bound_W
    assert not bad.any(), f"grad_weight: {bad.sum()} elements out, worst {np.abs(got_W - gW[cols])[bad].max():.3g}"


def test_fused_linear_out_of_range_idx_is_flagged():
    """The row's logp is NaN and the error bit is set; with beta > 0 its row factor is NaN
    too, so its dlogits and hidden-state gradient are NaN (with beta = 0 and no old_logp
    the policy-gradient factor of a NaN ratio is 0, as in grpo_loss_fused)."""
    pb = problem(1, 8, 32, 256, seed=3, beta=0.04, masked=False, zero_adv=False)
    pb["idx"][3] = 256
    out, err = run_gpu(pb, 4)
    assert err & rp.GRPO_DEVERR_IDX_OUT_OF_RANGE
    assert torch.isnan(out["logp"][3]) and torch.isnan(out["grad_hidden"][3]).all()
    assert not torch.isnan(out["grad_hidden"][2]).any()
