"""Vocabulary-parallel form on one GPU: the vocabulary is cut into shards (column views
of the full logits), each shard runs grpo_vocab_shard_stats, the statistics are stacked in
shard order (what an all-gather over the ranks returns), grpo_vocab_combine merges them,
and each shard's backward writes its columns of dlogits.  The result must be the full
rows' result: compared with the oracle on every row, and with the unsplit CUDA path.
"""

import numpy as np
import pytest
import torch

import oracle
from parity_util import assert_grad_rows, assert_plus_zero, assert_scalar_close, f32, rows_f64
from test_parity_gpu import (check_entropy_grad, compare_grpo_rows, edge_inputs, near_logp_inputs, oracle_logp,
                             run_gpu_grpo, select_rows)
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


def shard_views(x, starts):
    return [x[..., starts[k]:starts[k + 1]] for k in range(len(starts) - 1)]


def sharded_grpo(inp, starts, old, ref, T, beta, el, eh, with_entropy=True):
    """Shard statistics -> stacked in shard order -> combine -> per-shard backward."""
    B, L = inp.spec.B, inp.spec.L
    V = starts[-1]
    t = lambda a: None if a is None else torch.as_tensor(a, dtype=torch.float32).to(DEV)
    old_t, ref_t = t(old), t(ref)
    dev_err = torch.zeros(1, dtype=torch.int32, device=DEV)
    stats = torch.stack([rp.grpo_vocab_shard_stats(v, s, T=T, idx=inp.idx, mask=inp.mask)
                         for v, s in zip(shard_views(inp.logits, starts), starts)])
    f = rp.grpo_vocab_combine(stats, starts, B, L, T=T, idx=inp.idx, adv=inp.adv, grpo=True, beta=beta,
                              eps_low=el, eps_high=eh, old_logp=old_t, ref_logp=ref_t, mask=inp.mask,
                              with_entropy=with_entropy, dev_err=dev_err)
    dl = torch.empty(inp.logits.shape, dtype=inp.logits.dtype, device=DEV)
    for k, (v, s) in enumerate(zip(shard_views(inp.logits, starts), starts)):
        rp.grpo_loss_bwd_vocab_shard(v, s, V, inp.idx, inp.adv, inp.dloss, f["logp"], f["lse"], f["p_rest"],
                                     T=T, beta=beta, eps_low=el, eps_high=eh, old_logp=old_t, ref_logp=ref_t,
                                     mask=inp.mask, dlogits=dl[..., starts[k]:starts[k + 1]], dev_err=dev_err)
    torch.cuda.synchronize()
    return f, dl, int(dev_err.item()), stats


def oracle_p_rest(x_rows, idx, starts, T):
    """Mass of each row outside the shard that holds idx (from the oracle's softmax)."""
    z, lse = oracle.log_softmax_rows(x_rows, T)
    p = np.exp(z - lse[:, None])
    out = np.empty(len(idx))
    for r, i in enumerate(idx):
        k = np.searchsorted(starts, i, side="right") - 1
        out[r] = p[r].sum() - p[r, starts[k]:starts[k + 1]].sum()
    return out


@pytest.mark.parametrize("name,starts_of", [
    ("tiny_fp32", lambda V: [0, V]),                                   # one shard
    ("tiny_fp32", lambda V: [0, 100, 101, 333, V]),                    # a one-column shard
    ("grpo_b4_l512_v32000", lambda V: [0, 8000, 16000, 24000, V]),     # the pages' workload, 4 ranks
    ("grpo_b4_l512_v32000", lambda V: [0, 12345, 20001, V]),           # uneven, unaligned starts
])
def test_sharded_grpo_matches_oracle_and_unsplit(name, starts_of):
    spec = W.get(name)
    inp = W.generate(spec, 0, device=DEV)
    starts = starts_of(spec.V)
    T, beta, el, eh = f32(spec.T), f32(spec.beta), f32(spec.eps_low), f32(spec.eps_high)
    lp = oracle_logp(inp.logits, inp.idx.cpu().numpy(), T)
    old, ref = near_logp_inputs(inp, lp)
    f, dl, err, _ = sharded_grpo(inp, starts, old, ref, T, beta, el, eh)
    assert err == 0
    R = spec.rows
    rows = np.arange(R) if R <= 512 else np.unique(np.random.default_rng(1).integers(0, R, 160))
    compare_grpo_rows(inp, f, dl, rows, old, ref, T, beta, el, eh, f"sharded {name} {len(starts) - 1}")

    # p_rest against the oracle's softmax on the unmasked sampled rows
    live = rows if inp.mask is None else rows[inp.mask.cpu().numpy()[rows] != 0]
    xo = rows_f64(select_rows(inp.logits, live))
    o_rest = oracle_p_rest(xo, inp.idx.cpu().numpy()[live], np.asarray(starts), T)
    got = f["p_rest"][torch.from_numpy(live).to(DEV)].double().cpu().numpy()
    assert np.all(np.abs(got - o_rest) <= 1e-5 * o_rest + 1e-7), "p_rest"

    # the unsplit CUDA path: same zero rows bit for bit, scalars within the parity tolerance
    fu, dlu, _ = run_gpu_grpo(inp, old, ref, T, beta, el, eh)
    for k in ("loss", "logp", "lse", "entropy"):
        assert_scalar_close(f[k], fu[k].double().cpu().numpy(), f"sharded vs unsplit {k}")
    zs = (dl.reshape(R, -1).view(torch.int16 if dl.dtype == torch.bfloat16 else torch.int32) == 0).all(dim=1)
    zu = (dlu.reshape(R, -1).view(torch.int16 if dlu.dtype == torch.bfloat16 else torch.int32) == 0).all(dim=1)
    assert torch.equal(zs, zu)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("V,starts", [(9, [0, 4, 9]), (513, [0, 1, 256, 513]), (4097, [0, 1000, 2049, 3001, 4097])])
def test_sharded_edge_shapes_every_row(dtype, V, starts):
    """Misaligned rows, masked rows, a zero-advantage sequence, beta > 0."""
    B, L = 2, 5
    x, idx, adv, mask, dloss = edge_inputs(B, L, V, dtype, 3, 1, V * 11)
    inp = W.Inputs(W.get("tiny_fp32", B=B, L=L, V=V), x, idx, adv, mask, dloss, None, None, None, None)
    T, beta, el, eh = f32(0.8), f32(0.05), f32(0.2), f32(0.28)
    xo = rows_f64(select_rows(x, np.arange(B * L)))
    lp, _ = oracle.selective_log_softmax(xo, idx.cpu().numpy(), T)
    g = torch.Generator().manual_seed(V)
    old = oracle.round_to_fp32(lp + torch.randn(B * L, generator=g).double().numpy() * 0.3)
    ref = oracle.round_to_fp32(lp + torch.randn(B * L, generator=g).double().numpy() * 0.1)
    f, dl, err, stats = sharded_grpo(inp, starts, old, ref, T, beta, el, eh)
    assert err == 0
    compare_grpo_rows(inp, f, dl, np.arange(B * L), old, ref, T, beta, el, eh, f"sharded edge V={V}")
    masked = torch.nonzero(mask == 0)[:, 0]
    if len(masked):
        assert_plus_zero(stats[:, masked], "masked rows' shard statistics")
        assert_plus_zero(f["p_rest"][masked], "masked rows' p_rest")


def test_sharded_selective_log_softmax_and_entropy():
    """The selective-log-softmax form (combine without GRPO terms, shard backward with an
    upstream dlogp) and the entropy backward on shards with the full rows' lse and H."""
    B, L, V = 3, 7, 3001
    starts = [0, 1000, 1001, 2500, V]
    x, idx, _, _, _ = edge_inputs(B, L, V, torch.bfloat16, 1, 3, 5)
    R = B * L
    T = 1.3
    stats = torch.stack([rp.grpo_vocab_shard_stats(v, s, T=T, idx=idx) for v, s in zip(shard_views(x, starts), starts)])
    f = rp.grpo_vocab_combine(stats, starts, B, L, T=T, idx=idx)
    up = torch.randn(R, generator=torch.Generator().manual_seed(3)).float()
    up[2] = 0.0
    up = up.to(DEV)
    dl = torch.empty(x.shape, dtype=x.dtype, device=DEV)
    dH = torch.empty(x.shape, dtype=x.dtype, device=DEV)
    dent = torch.full((R,), -0.01, device=DEV)
    for k, (v, s) in enumerate(zip(shard_views(x, starts), starts)):
        rp.selective_log_softmax_bwd_vocab_shard(v, s, V, idx, up, f["lse"], f["p_rest"], T=T,
                                                 dlogits=dl[..., starts[k]:starts[k + 1]])
        rp.entropy_from_logits_bwd(v, dent, f["lse"], f["entropy"], T=T, dlogits=dH[..., starts[k]:starts[k + 1]])
    torch.cuda.synchronize()
    xo = rows_f64(select_rows(x, np.arange(R)))
    o_lp, o_lse = oracle.selective_log_softmax(xo, idx.cpu().numpy(), T)
    assert_scalar_close(f["logp"], o_lp, "sharded logp")
    assert_scalar_close(f["lse"], o_lse, "sharded lse")
    assert_scalar_close(f["entropy"], oracle.entropy_from_logits(xo, T), "sharded entropy")
    odl, og = oracle.selective_log_softmax_bwd(xo, idx.cpu().numpy(), up.double().cpu().numpy(), T)
    assert_grad_rows(dl.reshape(R, V), odl, og, np.zeros(R, bool), "sharded slsm dlogits")
    check_entropy_grad(dH.reshape(R, V), xo, np.full(R, -0.01), T, f["entropy"].cpu().numpy(),
                       f["lse"].cpu().numpy(), "sharded entropy bwd")

    # entropy / lse only: no idx
    g = rp.grpo_vocab_combine(stats, starts, B, L, T=T)
    assert torch.equal(g["lse"], f["lse"]) and torch.equal(g["entropy"], f["entropy"])


def test_sharded_out_of_range_idx_is_flagged():
    B, L, V = 1, 4, 640
    starts = [0, 320, V]
    x, idx, adv, _, dloss = edge_inputs(B, L, V, torch.float32, 0, 0, 9)
    adv[:] = 1.0
    idx[1] = V          # past the last shard
    idx[2] = -1
    inp = W.Inputs(W.get("tiny_fp32", B=B, L=L, V=V), x, idx, adv, None, dloss.abs() + 0.1, None, None, None, None)
    f, dl, err, _ = sharded_grpo(inp, starts, None, None, 1.0, 0.0, 0.2, 0.2)
    assert err & rp.GRPO_DEVERR_IDX_OUT_OF_RANGE
    for k in ("logp", "loss", "p_rest"):
        assert torch.isnan(f[k][1]) and torch.isnan(f[k][2]) and not torch.isnan(f[k][0]), k
    assert torch.isnan(dl[0, 1]).all() and torch.isnan(dl[0, 2]).all() and not torch.isnan(dl[0, 0]).any()
