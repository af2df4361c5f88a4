"""The torch.autograd wrappers: the same numbers as the C-ABI calls they marshal, and the
oracle's gradients through ``.backward()`` (GPU)."""

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from parity_util import assert_grad_rows, assert_scalar_close, f32, rows_f64
from test_parity_gpu import check_entropy_grad, compare_grpo_rows, near_logp_inputs, oracle_logp
from rl_fine_tuning_pass_gb300 import autograd as ag
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


def same_bits(a: torch.Tensor, b: torch.Tensor, what: str):
    assert a.shape == b.shape and a.dtype == b.dtype, what
    assert torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8)), what


@pytest.mark.parametrize("name,seed", [("tiny_fp32", 0), ("tiny_fp32", 1), ("grpo_b4_l512_v32000", 0)])
def test_grpo_loss_backward_is_the_capi_backward(name, seed):
    """(loss * w).sum().backward() gives grpo_loss_bwd with dloss = w, bit for bit, and the
    oracle's gradient on every row of the tiny case (sampled rows of the pages' workload)."""
    spec = W.get(name)
    inp = W.generate(spec, seed, device=DEV)
    T, beta, el, eh = f32(spec.T), f32(spec.beta), f32(spec.eps_low), f32(spec.eps_high)
    lp = oracle_logp(inp.logits, inp.idx.cpu().numpy(), T)
    old, ref = near_logp_inputs(inp, lp)
    t = lambda a: None if a is None else torch.as_tensor(a, dtype=torch.float32).to(DEV)
    old_t, ref_t = t(old), t(ref)
    w = inp.dloss

    x = inp.logits.detach().requires_grad_(True)   # same addresses as the direct calls below
    loss, aux = ag.grpo_loss(x, inp.idx, inp.adv, T=T, beta=beta, eps_low=el, eps_high=eh, old_logp=old_t,
                             ref_logp=ref_t, mask=inp.mask)
    (loss * w).sum().backward()
    torch.cuda.synchronize()

    f = rp.grpo_loss_fwd(inp.logits, inp.idx, inp.adv, T=T, beta=beta, eps_low=el, eps_high=eh, old_logp=old_t,
                         ref_logp=ref_t, mask=inp.mask, with_entropy=True)
    dl = rp.grpo_loss_bwd(inp.logits, inp.idx, inp.adv, w, f["logp"], f["lse"], T=T, beta=beta, eps_low=el,
                          eps_high=eh, old_logp=old_t, ref_logp=ref_t, mask=inp.mask)
    torch.cuda.synchronize()
    same_bits(loss.detach(), f["loss"], "loss")
    for k in ("logp", "kl", "is_clipped", "entropy"):
        same_bits(aux[k], f[k], k)
        assert not aux[k].requires_grad
    same_bits(x.grad, dl, "logits.grad")

    out = dict(f)
    out["loss"] = loss.detach()
    rows = (np.arange(spec.rows) if spec.rows <= 64 else
            np.unique(np.random.default_rng(seed).integers(0, spec.rows, 96)))
    compare_grpo_rows(dataclasses.replace(inp, dloss=w), out, x.grad, rows, old, ref, T, beta, el, eh,
                      f"autograd {name} s{seed}")


def test_loss_plus_entropy_bonus_accumulates_both_gradients():
    """loss.sum() - c * H.sum(): autograd adds the two C-ABI backwards (fp32, same addition)."""
    spec = W.get("tiny_fp32")
    inp = W.generate(spec, 3, device=DEV)
    T, c = 0.8, 0.01
    x = inp.logits.detach().requires_grad_(True)
    loss, _ = ag.grpo_loss(x, inp.idx, inp.adv, T=T, beta=0.0, eps_low=0.2, eps_high=0.28)
    H = ag.entropy(x, T=T)
    (loss.sum() - c * H.sum()).backward()

    f = rp.grpo_loss_fwd(inp.logits, inp.idx, inp.adv, T=T, beta=0.0, eps_low=0.2, eps_high=0.28)
    ones = torch.ones(spec.rows, dtype=torch.float32, device=DEV)
    d1 = rp.grpo_loss_bwd(inp.logits, inp.idx, inp.adv, ones, f["logp"], f["lse"], T=T, beta=0.0, eps_low=0.2,
                          eps_high=0.28)
    H2, lse = rp.entropy_from_logits(inp.logits, T=T, return_lse=True)
    d2 = rp.entropy_from_logits_bwd(inp.logits, torch.full((spec.rows,), -c, device=DEV), lse, H2, T=T)
    torch.cuda.synchronize()
    same_bits(H.detach(), H2, "entropy")
    # autograd sums the two gradient tensors in the order their nodes finish; either order
    # of an fp32 addition of two values is the same number
    same_bits(x.grad, d1 + d2, "accumulated logits.grad")
    xo = rows_f64(inp.logits.reshape(-1, spec.V))
    o1, g1 = oracle.grpo_loss_bwd(xo, inp.idx.cpu().numpy(), None, None, oracle.per_row(inp.adv.cpu().numpy(), spec.L),
                                  None, np.ones(spec.rows), T, 0.0, 0.2, 0.28)
    assert_grad_rows(d1.reshape(-1, spec.V), o1, g1, np.zeros(spec.rows, bool), "grpo term of the sum")
    check_entropy_grad(d2.reshape(-1, spec.V), xo, np.full(spec.rows, -c), T, H2.cpu().numpy(), lse.cpu().numpy(),
                       "entropy term of the sum")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_selective_log_softmax_autograd_on_a_shifted_view(dtype):
    """The usual logits[:, :-1, :] view: gradient lands in the base tensor's rows, last
    position of every sequence zero, and equals selective_log_softmax_bwd on the view."""
    B, L, V = 3, 40, 1000
    g = torch.Generator().manual_seed(7)
    full = (torch.randn(B, L + 1, V, generator=g) * 2).to(torch.bfloat16 if dtype == "bf16" else torch.float32)
    full = full.to(DEV).requires_grad_(True)
    view = full[:, :-1, :]
    idx = torch.randint(0, V, (B * L,), generator=g).to(DEV)
    up = torch.randn(B * L, generator=g).float().to(DEV)
    T = 1.3
    logp = ag.selective_log_softmax(view, idx, T=T)
    (logp * up).sum().backward()
    torch.cuda.synchronize()

    lp2, lse = rp.selective_log_softmax_fwd(view.detach(), idx, T=T)
    dl = rp.selective_log_softmax_bwd(view.detach(), idx, up, lse, T=T)
    torch.cuda.synchronize()
    same_bits(logp.detach(), lp2, "logp")
    same_bits(full.grad[:, :-1, :].contiguous(), dl, "view grad")
    assert torch.count_nonzero(full.grad[:, -1, :]) == 0

    xo = rows_f64(view.detach().reshape(-1, V))
    o_lp, _ = oracle.selective_log_softmax(xo, idx.cpu().numpy(), T)
    assert_scalar_close(logp.detach(), o_lp, "autograd slsm logp")
    odl, og = oracle.selective_log_softmax_bwd(xo, idx.cpu().numpy(), up.double().cpu().numpy(), T)
    assert_grad_rows(dl.reshape(-1, V), odl, og, np.zeros(B * L, bool), "autograd slsm dlogits")
