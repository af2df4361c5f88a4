"""CUDA path vs the fp64 oracle on the same seeded inputs (GPU).

Every call goes through the C ABI (ctypes binding).  Small workloads are compared on
every row; the large ones (V = 32000 with 65536 rows, V = 151936) run at full size in
the launch configuration the benchmark times and are compared on sampled rows, plus
whole-tensor properties (bit-exact zero rows, entropy bounds, row sums).
Tolerances are documented in parity_util.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from parity_util import (ambiguous_rows, assert_bf16_grad_close, assert_grad_rows, assert_plus_zero,
                         assert_scalar_close, bf16_bits, f32, row_error_budget, rows_f64)
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


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def select_rows(logits: torch.Tensor, rows: np.ndarray) -> torch.Tensor:
    B, L, V = logits.shape
    r = torch.from_numpy(np.asarray(rows, dtype=np.int64)).to(logits.device)
    return logits[r // L, r % L]


def oracle_logp(logits, idx_np, T, chunk=256, rows=None):
    """The oracle's logp of `rows` (default: every row), in chunks of rows."""
    B, L, V = logits.shape
    rows = np.arange(B * L) if rows is None else np.asarray(rows)
    out = np.empty(len(rows))
    for k0 in range(0, len(rows), chunk):
        part = rows[k0:k0 + chunk]
        lp, _ = oracle.selective_log_softmax(rows_f64(select_rows(logits, part)), idx_np[part], T)
        out[k0:k0 + len(part)] = lp
    return out


def torch_logp(logits, idx, T, chunk=1024):
    """log_softmax(x / T)[idx] with plain torch ops (used only to place old/ref near logp
    on rows that the oracle does not check)."""
    B, L, V = logits.shape
    flat = logits.reshape(B * L, V)
    out = torch.empty(B * L, dtype=torch.float32, device=logits.device)
    for r0 in range(0, B * L, chunk):
        xs = flat[r0:r0 + chunk].float() / T
        out[r0:r0 + chunk] = torch.log_softmax(xs, dim=-1).gather(1, idx[r0:r0 + chunk, None])[:, 0]
    return out


def near_logp_inputs(inp, logp_np):
    """old/ref = logp + the generator's offsets, rounded to fp32 (numpy, host)."""
    old = ref = None
    if inp.old_offset is not None:
        old = oracle.round_to_fp32(logp_np + inp.old_offset.cpu().numpy().astype(np.float64))
    if inp.ref_offset is not None:
        ref = oracle.round_to_fp32(logp_np + inp.ref_offset.cpu().numpy().astype(np.float64))
    return old, ref


def run_gpu_grpo(inp, old, ref, T, beta, el, eh, dlogits=None):
    dev_err = torch.zeros(1, dtype=torch.int32, device=DEV)
    t = lambda a: None if a is None else torch.as_tensor(a, dtype=torch.float32).to(DEV)
    old_t, ref_t = t(old), t(ref)
    f = rp.grpo_loss_fwd(inp.logits, inp.idx, inp.adv, T=T, beta=beta, eps_low=el, eps_high=eh,
                         old_logp=old_t, ref_logp=ref_t, mask=inp.mask, with_entropy=True, dev_err=dev_err)
    dl = rp.grpo_loss_bwd(inp.logits, inp.idx, inp.adv, inp.dloss, f["logp"], f["lse"], T=T, beta=beta,
                          eps_low=el, eps_high=eh, old_logp=old_t, ref_logp=ref_t, mask=inp.mask,
                          dlogits=dlogits, dev_err=dev_err)
    torch.cuda.synchronize()
    return f, dl, int(dev_err.item())


def compare_grpo_rows(inp, f, dl, rows, old, ref, T, beta, el, eh, tag):
    """Oracle on `rows` vs the GPU outputs on those rows; returns the oracle g."""
    L = inp.spec.L
    x = rows_f64(select_rows(inp.logits, rows))
    idx = inp.idx.cpu().numpy()[rows]
    adv = oracle.per_row(inp.adv.cpu().numpy(), L)[rows]
    mask = None if inp.mask is None else inp.mask.cpu().numpy()[rows]
    dloss = inp.dloss.cpu().numpy().astype(np.float64)[rows]
    o_old = None if old is None else np.asarray(old, dtype=np.float64)[rows]
    o_ref = None if ref is None else np.asarray(ref, dtype=np.float64)[rows]
    of = oracle.grpo_loss_fwd(x, idx, o_old, o_ref, adv, mask, T, beta, el, eh)
    odl, g = oracle.grpo_loss_bwd(x, idx, o_old, o_ref, adv, mask, dloss, T, beta, el, eh)
    r_t = torch.from_numpy(rows).to(DEV)
    dlogp = f["logp"][r_t].double().cpu().numpy() - of["logp"]
    dlse = f["lse"][r_t].double().cpu().numpy() - of["lse"]
    rho = row_error_budget(g, of["ratio"], adv, beta, of["logp"], o_ref, dloss, T, dlogp, dlse)
    amb = ambiguous_rows(of["ratio"], adv, mask, el, eh, rho)
    for k in ("loss", "logp", "lse", "kl", "entropy"):
        assert_scalar_close(f[k][r_t], of[k], f"{tag} {k}")
    masked = np.zeros(len(rows), bool) if mask is None else (mask == 0)
    for k in ("loss", "logp", "lse", "kl", "entropy"):
        if np.any(masked):
            assert_plus_zero(f[k][r_t][torch.from_numpy(masked).to(DEV)], f"{tag} masked {k}")
    clip_gpu = f["is_clipped"][r_t].cpu().numpy().astype(bool)
    assert np.array_equal(clip_gpu[~amb], of["is_clipped"][~amb]), f"{tag} is_clipped"
    assert amb.sum() <= max(2, 0.01 * len(rows)), f"{tag}: {amb.sum()} ambiguous rows"
    assert_grad_rows(select_rows(dl, rows), odl, g, amb, f"{tag} dlogits", rho=rho)
    return g, amb


# ---------------------------------------------------------------------------
# the tiny fp32 case and the pages' GRPO backward workload, every row
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_fp32_grpo_every_row(seed):
    spec = W.get("tiny_fp32")
    inp = W.generate(spec, seed, device=DEV)
    T, beta, el, eh = f32(spec.T), f32(spec.beta), f32(spec.eps_low), f32(spec.eps_high)
    lp = oracle_logp(inp.logits, inp.idx.cpu().numpy(), T)
    old, ref = near_logp_inputs(inp, lp)
    f, dl, err = run_gpu_grpo(inp, old, ref, T, beta, el, eh)
    assert err == 0
    compare_grpo_rows(inp, f, dl, np.arange(spec.rows), old, ref, T, beta, el, eh, f"tiny s{seed}")


@pytest.mark.parametrize("seed", [0, 1])
def test_tiny_fp32_slsm_and_entropy_every_row(seed):
    spec = W.get("tiny_fp32")
    inp = W.generate(spec, seed, device=DEV)
    T = 0.7
    x = rows_f64(inp.logits.reshape(-1, spec.V))
    idx = inp.idx.cpu().numpy()
    logp, lse = rp.selective_log_softmax_fwd(inp.logits, inp.idx, T=T)
    H = rp.entropy_from_logits(inp.logits, T=T)
    up = torch.randn(spec.rows, generator=torch.Generator().manual_seed(seed)).float()
    up[3] = 0.0
    up[5] = -0.0
    dl = rp.selective_log_softmax_bwd(inp.logits, inp.idx, up.to(DEV), lse, T=T)
    torch.cuda.synchronize()
    o_lp, o_lse = oracle.selective_log_softmax(x, idx, T)
    assert_scalar_close(logp, o_lp, "slsm logp")
    assert_scalar_close(lse, o_lse, "slsm lse")
    assert_scalar_close(H, oracle.entropy_from_logits(x, T), "entropy")
    odl, g = oracle.selective_log_softmax_bwd(x, idx, up.double().numpy(), T)
    assert_grad_rows(dl.reshape(-1, spec.V), odl, g, np.zeros(spec.rows, bool), "slsm dlogits")


def test_pages_grpo_workload_every_row():
    """B=4, L=512, V=32000 bf16, beta=0, half the sequences with A == 0, 10% padding."""
    spec = W.get("grpo_b4_l512_v32000")
    inp = W.generate(spec, 0, device=DEV)
    T, beta, el, eh = f32(spec.T), 0.0, f32(spec.eps_low), f32(spec.eps_high)
    lp = oracle_logp(inp.logits, inp.idx.cpu().numpy(), T)
    old, ref = near_logp_inputs(inp, lp)
    f, dl, err = run_gpu_grpo(inp, old, ref, T, beta, el, eh)
    assert err == 0
    gs = []
    for r0 in range(0, spec.rows, 256):
        g, _ = compare_grpo_rows(inp, f, dl, np.arange(r0, r0 + 256), old, ref, T, beta, el, eh, "pages c2")
        gs.append(g)
    g = np.concatenate(gs)
    zero_frac = float(np.mean(g == 0.0))
    # 2 of 4 sequences have A == 0, 10% padding, plus clipped tokens with beta == 0
    assert 0.55 < zero_frac < 0.65, zero_frac
    assert np.any((g == 0) & (oracle.per_row(inp.adv.cpu().numpy(), spec.L) != 0)
                  & (inp.mask.cpu().numpy() == 1)), "no clipped zero rows in the workload"


# ---------------------------------------------------------------------------
# large workloads: sampled rows + whole-tensor properties
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("strided", [False, True], ids=["contiguous", "view_of_L_plus_1"])
def test_entropy_slsm_v32000_full_size(strided):
    spec = W.get("entropy_slsm_b16_l4096_v32000", strided=strided)
    inp = W.generate(spec, 0, device=DEV)
    T = f32(spec.T)
    H = rp.entropy_from_logits(inp.logits, T=T)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    logp, lse = rp.selective_log_softmax_fwd(inp.logits, inp.idx, T=T, dev_err=err)
    dl = rp.selective_log_softmax_bwd(inp.logits, inp.idx, inp.upstream, lse, T=T, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # whole tensor: 0 <= H <= ln V, lse >= max x / T, row sums ~ 0
    assert float(H.min()) >= -1e-5 and float(H.max()) <= math.log(spec.V) + 1e-4
    xmax = inp.logits.float().amax(dim=-1).reshape(-1) / T
    assert bool(torch.all(lse >= xmax - 1e-4))
    rs = dl.float().sum(dim=-1).reshape(-1).abs()
    assert float(rs.max()) <= (1.0 / spec.rows / T) * spec.V * 2.0 ** -8
    # sampled rows, including peaked ones
    peaked = torch.nonzero(inp.logits.float().amax(dim=-1).reshape(-1) > 14.0)[:, 0].cpu().numpy()
    rows = np.unique(np.concatenate([W.sample_rows(spec.rows, 40, 1), peaked[::max(1, len(peaked) // 24)]]))
    x = rows_f64(select_rows(inp.logits, rows))
    idx = inp.idx.cpu().numpy()[rows]
    o_lp, o_lse = oracle.selective_log_softmax(x, idx, T)
    r_t = torch.from_numpy(rows).to(DEV)
    assert_scalar_close(logp[r_t], o_lp, "slsm logp")
    assert_scalar_close(lse[r_t], o_lse, "slsm lse")
    assert_scalar_close(H[r_t], oracle.entropy_from_logits(x, T), "entropy")
    odl, g = oracle.selective_log_softmax_bwd(x, idx, inp.upstream.cpu().numpy()[rows], T)
    assert_grad_rows(select_rows(dl, rows), odl, g, np.zeros(len(rows), bool), "slsm dlogits")


def _sampled_grpo(spec, inp, T, beta, el, eh, n_rows, seed, dlogits=None):
    """old/ref from torch's log-softmax on all rows, and from the oracle on the sampled rows."""
    rows = W.sample_rows(spec.rows, n_rows, seed)
    lp_all = torch_logp(inp.logits, inp.idx, T).double().cpu().numpy()
    lp_all[rows] = oracle.selective_log_softmax(rows_f64(select_rows(inp.logits, rows)),
                                                inp.idx.cpu().numpy()[rows], T)[0]
    old, ref = near_logp_inputs(inp, lp_all)
    f, dl, err = run_gpu_grpo(inp, old, ref, T, beta, el, eh, dlogits=dlogits)
    assert err == 0
    g, _ = compare_grpo_rows(inp, f, dl, rows, old, ref, T, beta, el, eh, spec.name)
    return f, dl, rows, g


def test_qwen3_head_grpo_full_size():
    spec = W.get("grpo_qwen3_b16_l1024_v151936")
    inp = W.generate(spec, 0, device=DEV)
    T, beta, el, eh = f32(spec.T), f32(spec.beta), f32(spec.eps_low), f32(spec.eps_high)
    f, dl, rows, g = _sampled_grpo(spec, inp, T, beta, el, eh, 40, 3)
    masked = inp.mask == 0
    assert bool(masked.any())
    assert_plus_zero(dl.reshape(-1, spec.V)[masked], "masked dlogits rows")
    for k in ("loss", "logp", "lse", "kl", "entropy"):
        assert_plus_zero(f[k][masked], f"masked {k}")
    live = ~masked
    assert float(f["entropy"][live].min()) > 0.0 and float(f["entropy"][live].max()) <= math.log(spec.V) + 1e-4


@pytest.fixture(scope="module")
def sweep_inputs():
    spec = W.get("sweep_b16_l4096_v151936")
    inp = W.generate(spec, 0, device=DEV)
    dl = torch.empty_like(inp.logits)
    yield spec, inp, dl
    del inp, dl
    torch.cuda.empty_cache()


@pytest.mark.parametrize("beta", [0.0, 0.04])
@pytest.mark.parametrize("zero_seqs", [0, 4, 8, 12, 16])
def test_sweep_v151936_full_size(sweep_inputs, beta, zero_seqs):
    spec0, inp0, dl = sweep_inputs
    spec = spec0.with_(beta=beta, zero_adv_seqs=zero_seqs)
    adv = W._advantages(spec, 0).to(DEV)
    inp = W.Inputs(spec, inp0.logits, inp0.idx, adv, inp0.mask, inp0.dloss, inp0.old_offset,
                   inp0.ref_offset, inp0.upstream, inp0.lengths)
    T, el, eh = f32(spec.T), f32(spec.eps_low), f32(spec.eps_high)
    f, dl, rows, g = _sampled_grpo(spec, inp, T, f32(beta), el, eh, 12, 5 + zero_seqs, dlogits=dl)
    zero_seq = torch.nonzero(adv == 0)[:, 0]
    assert len(zero_seq) == zero_seqs
    if beta == 0.0 and zero_seqs:
        assert_plus_zero(dl[zero_seq], "zero-advantage sequences with beta=0")
    if beta != 0.0 and zero_seqs:
        # zero advantage no longer gives zero rows: the KL term keeps a gradient
        assert bool((dl[zero_seq[0], :64].float() != 0).any())


# ---------------------------------------------------------------------------
# edge cases: ragged V, misaligned and odd-strided rows, aliasing, special values
# ---------------------------------------------------------------------------

def strided_logits(B, L, V, dtype, offset, extra, seed, scale=2.0):
    """[B, L, V] view into a larger buffer: rows start `offset` elements in, row stride
    V + extra (so starts are generally not 16-byte aligned)."""
    g = torch.Generator().manual_seed(seed)
    sl = V + extra
    n = offset + B * L * sl + 8
    buf = (torch.randn(n, generator=g) * scale).to(dtype).to(DEV)
    return torch.as_strided(buf, (B, L, V), (L * sl, sl, 1), offset), buf


def edge_inputs(B, L, V, dtype, offset, extra, seed):
    x, _ = strided_logits(B, L, V, dtype, offset, extra, seed)
    g = torch.Generator().manual_seed(seed + 1)
    R = B * L
    idx = torch.randint(0, V, (R,), generator=g)
    adv = torch.randn(B, generator=g).float()
    adv[0] = 0.0
    mask = (torch.rand(R, generator=g) > 0.25).to(torch.uint8)
    dloss = (torch.rand(R, generator=g) + 0.1).float() * mask.float()
    return x, idx.to(DEV), adv.to(DEV), mask.to(DEV), dloss.to(DEV)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("V", [1, 2, 7, 8, 9, 15, 16, 17, 100, 511, 512, 513, 4097, 8191, 40000])
@pytest.mark.parametrize("offset,extra", [(0, 0), (1, 3), (3, 1)])
def test_edge_shapes_every_row(dtype, V, offset, extra):
    B, L = 2, 5
    R = B * L
    seed = V * 7 + offset
    x, idx, adv, mask, dloss = edge_inputs(B, L, V, dtype, offset, extra, seed)
    T, beta, el, eh = f32(0.8), f32(0.05), f32(0.2), f32(0.28)
    xo = rows_f64(select_rows(x, np.arange(R)))
    idx_np = idx.cpu().numpy()
    lp, _ = oracle.selective_log_softmax(xo, idx_np, T)
    g = torch.Generator().manual_seed(V)
    old = oracle.round_to_fp32(lp + torch.randn(R, generator=g).double().numpy() * 0.3)
    ref = oracle.round_to_fp32(lp + torch.randn(R, generator=g).double().numpy() * 0.1)
    inp = W.Inputs(W.get("tiny_fp32", B=B, L=L, V=V), x, idx, adv, mask, dloss, None, None, None, None)
    # out-of-phase dlogits: rows shifted by one element against the logits rows
    dl_buf = torch.empty(B * L * (V + 2) + 9, dtype=dtype, device=DEV)
    dl_view = torch.as_strided(dl_buf, (B, L, V), (L * (V + 2), V + 2, 1), 1 + offset)
    f, dl, err = run_gpu_grpo(inp, old, ref, T, beta, el, eh, dlogits=dl_view)
    assert err == 0
    compare_grpo_rows(inp, f, dl, np.arange(R), old, ref, T, beta, el, eh, f"edge V={V}")
    # in-place on an identical copy: bit-identical to an out-of-place run whose output rows
    # have the same layout (hence the same row split and summation order)
    x2, _ = strided_logits(B, L, V, dtype, offset, extra, seed)
    same_layout, _ = strided_logits(B, L, V, dtype, offset, extra, seed + 99)
    _, dl_same, err3 = run_gpu_grpo(inp, old, ref, T, beta, el, eh, dlogits=same_layout)
    inp2 = W.Inputs(inp.spec, x2, idx, adv, mask, dloss, None, None, None, None)
    _, dl2, err2 = run_gpu_grpo(inp2, old, ref, T, beta, el, eh, dlogits=x2)
    assert err2 == 0 and err3 == 0 and dl2.data_ptr() == x2.data_ptr()
    assert torch.equal(bf16_or_f32_bits(select_rows(dl2, np.arange(R))),
                       bf16_or_f32_bits(select_rows(dl_same, np.arange(R))))
    # selective log-softmax and entropy on the same misaligned rows
    H = rp.entropy_from_logits(x, T=T)
    slp, slse = rp.selective_log_softmax_fwd(x, idx, T=T)
    up = dloss.clone()
    sdl = rp.selective_log_softmax_bwd(x, idx, up, slse, T=T, dlogits=dl_view)
    torch.cuda.synchronize()
    o_lp, o_lse = oracle.selective_log_softmax(xo, idx_np, T)
    assert_scalar_close(slp, o_lp, "edge slsm logp")
    assert_scalar_close(slse, o_lse, "edge slsm lse")
    assert_scalar_close(H, oracle.entropy_from_logits(xo, T), "edge entropy")
    odl, og = oracle.selective_log_softmax_bwd(xo, idx_np, up.cpu().double().numpy(), T)
    assert_grad_rows(select_rows(sdl, np.arange(R)), odl, og, np.zeros(R, bool), f"edge slsm V={V}")


def bf16_or_f32_bits(t):
    t = t.contiguous()
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def test_masked_rows_ignore_their_idx_and_bad_idx_is_flagged():
    B, L, V = 1, 6, 300
    x, idx, adv, mask, dloss = edge_inputs(B, L, V, torch.bfloat16, 0, 0, seed=11)
    adv.fill_(1.0)
    mask[:] = torch.tensor([1, 0, 1, 0, 1, 1], dtype=torch.uint8)
    idx[1] = -100           # padding index on a masked row: never read
    idx[3] = V + 5
    idx[4] = V              # out of range on an unmasked row
    idx[5] = -1
    dloss.fill_(0.5)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    f = rp.grpo_loss_fwd(x, idx, adv, T=1.0, beta=0.0, eps_low=0.2, eps_high=0.2, mask=mask,
                         with_entropy=True, dev_err=err)
    dl = rp.grpo_loss_bwd(x, idx, adv, dloss, f["logp"], f["lse"], T=1.0, beta=0.0, eps_low=0.2,
                          eps_high=0.2, mask=mask, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == rp.GRPO_DEVERR_IDX_OUT_OF_RANGE
    for r in (4, 5):
        assert math.isnan(float(f["logp"][r])) and math.isnan(float(f["loss"][r]))
        assert math.isfinite(float(f["lse"][r])) and math.isfinite(float(f["entropy"][r]))
        assert bool(torch.isnan(dl[0, r].float()).all())
    for r in (1, 3):
        assert_plus_zero(dl[0, r], "masked row")
        assert float(f["loss"][r]) == 0.0
    assert math.isfinite(float(f["loss"][0])) and math.isfinite(float(f["loss"][2]))
    err.zero_()
    slp, _ = rp.selective_log_softmax_fwd(x, idx, T=1.0, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == rp.GRPO_DEVERR_IDX_OUT_OF_RANGE
    assert math.isnan(float(slp[1])) and math.isfinite(float(slp[0]))


def test_nan_and_inf_logits_propagate_like_the_oracle():
    V = 257
    x = (torch.randn(6, V, generator=torch.Generator().manual_seed(3)) * 2).float()
    x[1, 10] = float("nan")
    x[2, 20] = float("inf")
    x[3, :] = float("-inf")
    x[4, 30] = float("-inf")
    x[5, 40] = 1e8      # |x / T| below 2^30: the documented input range
    idx = torch.tensor([5, 6, 7, 8, 9, 40])
    xd, idd = x.to(DEV), idx.to(DEV)
    lp, lse = rp.selective_log_softmax_fwd(xd, idd, T=1.0)
    H = rp.entropy_from_logits(xd, T=1.0)
    torch.cuda.synchronize()
    xo = x.double().numpy()
    with np.errstate(all="ignore"):
        o_lp, o_lse = oracle.selective_log_softmax(xo, idx.numpy(), 1.0)
        o_H = oracle.entropy_from_logits(xo, 1.0)
    assert_scalar_close(lp, o_lp, "special logp")
    assert_scalar_close(lse, o_lse, "special lse")
    assert_scalar_close(H, o_H, "special entropy", atol=1e-4)


def test_spiked_rows_keep_one_minus_p_accurate():
    """p_idx close to 1: the idx element g (1 - p_idx) must still be within 1 bf16 ulp."""
    R, V = 8, 32000
    g = torch.Generator().manual_seed(5)
    x = (torch.randn(R, V, generator=g) * 3.0)
    idx = torch.randint(0, V, (R,), generator=g)
    x[torch.arange(R), idx] += torch.tensor([20., 24., 26., 28., 30., 33., 36., 40.])
    xb = x.to(torch.bfloat16).to(DEV)
    idd = idx.to(DEV)
    up = torch.full((R,), 0.37).to(DEV)
    lp, lse = rp.selective_log_softmax_fwd(xb, idd, T=1.0)
    dl = rp.selective_log_softmax_bwd(xb, idd, up, lse, T=1.0)
    torch.cuda.synchronize()
    xo = rows_f64(xb)
    odl, og = oracle.selective_log_softmax_bwd(xo, idx.numpy(), np.full(R, f32(0.37)), 1.0)
    assert_bf16_grad_close(bf16_bits(dl), odl, "spiked dlogits")
    assert_scalar_close(lp, oracle.selective_log_softmax(xo, idx.numpy(), 1.0)[0], "spiked logp")


def test_large_magnitude_and_temperature():
    R, V = 4, 5000
    x = torch.randn(R, V, generator=torch.Generator().manual_seed(9)) * 3e3
    xb = x.to(torch.bfloat16).to(DEV)
    idx = torch.randint(0, V, (R,), generator=torch.Generator().manual_seed(10)).to(DEV)
    for T in (0.05, 1.0, 7.5):
        lp, lse = rp.selective_log_softmax_fwd(xb, idx, T=T)
        H = rp.entropy_from_logits(xb, T=T)
        torch.cuda.synchronize()
        xo = rows_f64(xb)
        o_lp, o_lse = oracle.selective_log_softmax(xo, idx.cpu().numpy(), f32(T))
        assert_scalar_close(lse, o_lse, f"lse T={T}")
        assert_scalar_close(lp, o_lp, f"logp T={T}", atol=1e-5 * max(1.0, float(np.abs(o_lp).max()) * 0.1))
        assert_scalar_close(H, oracle.entropy_from_logits(xo, f32(T)), f"H T={T}", atol=1e-4)


def test_on_policy_and_sign_of_zero():
    """old_logp absent (ratio 1); upstream -0.0 and dloss -0.0 give +0.0 rows."""
    B, L, V = 2, 4, 1000
    x, idx, adv, mask, dloss = edge_inputs(B, L, V, torch.bfloat16, 0, 0, seed=21)
    mask.fill_(1)
    dloss[2] = -0.0
    inp = W.Inputs(W.get("tiny_fp32", B=B, L=L, V=V), x, idx, adv, mask, dloss, None, None, None, None)
    T = f32(1.3)
    f, dl, err = run_gpu_grpo(inp, None, None, T, 0.0, f32(0.2), f32(0.2))
    assert err == 0
    compare_grpo_rows(inp, f, dl, np.arange(B * L), None, None, T, 0.0, f32(0.2), f32(0.2), "on-policy")
    assert_plus_zero(dl[0, 2], "dloss = -0.0 row")
    up = torch.full((B * L,), -0.0, device=DEV)
    _, lse = rp.selective_log_softmax_fwd(x, idx, T=T)
    sdl = rp.selective_log_softmax_bwd(x, idx, up, lse, T=T)
    torch.cuda.synchronize()
    assert_plus_zero(sdl, "upstream -0.0")


def test_empty_inputs_launch_nothing():
    x = torch.empty(0, 7, 64, dtype=torch.bfloat16, device=DEV)
    idx = torch.empty(0, dtype=torch.int64, device=DEV)
    assert rp.entropy_from_logits(x).numel() == 0
    lp, lse = rp.selective_log_softmax_fwd(x, idx)
    assert lp.numel() == 0
    f = rp.grpo_loss_fwd(x, idx, torch.empty(0, device=DEV), T=1.0, beta=0.0, eps_low=0.2, eps_high=0.2)
    assert f["loss"].numel() == 0


# ---------------------------------------------------------------------------
# fused single-read forward + backward
# ---------------------------------------------------------------------------

def run_gpu_fused(inp, old, ref, T, beta, el, eh, dlogits=None):
    dev_err = torch.zeros(1, dtype=torch.int32, device=DEV)
    t = lambda a: None if a is None else torch.as_tensor(a, dtype=torch.float32).to(DEV)
    f = rp.grpo_loss_fused(inp.logits, inp.idx, inp.adv, inp.dloss, T=T, beta=beta, eps_low=el, eps_high=eh,
                           old_logp=t(old), ref_logp=t(ref), mask=inp.mask, with_entropy=True, dlogits=dlogits,
                           dev_err=dev_err)
    torch.cuda.synchronize()
    return f, f["dlogits"], int(dev_err.item())


@pytest.mark.parametrize("seed", [0, 1])
def test_fused_tiny_fp32_every_row(seed):
    spec = W.get("tiny_fp32")
    inp = W.generate(spec, seed, device=DEV)
    T, beta, el, eh = f32(spec.T), f32(spec.beta), f32(spec.eps_low), f32(spec.eps_high)
    lp = oracle_logp(inp.logits, inp.idx.cpu().numpy(), T)
    old, ref = near_logp_inputs(inp, lp)
    f, dl, err = run_gpu_fused(inp, old, ref, T, beta, el, eh)
    assert err == 0
    compare_grpo_rows(inp, f, dl, np.arange(spec.rows), old, ref, T, beta, el, eh, f"fused tiny s{seed}")


def test_fused_pages_workload_every_row_and_matches_separate():
    spec = W.get("grpo_b4_l512_v32000")
    inp = W.generate(spec, 0, device=DEV)
    T, beta, el, eh = f32(spec.T), 0.0, f32(spec.eps_low), f32(spec.eps_high)
    lp = oracle_logp(inp.logits, inp.idx.cpu().numpy(), T)
    old, ref = near_logp_inputs(inp, lp)
    f, dl, err = run_gpu_fused(inp, old, ref, T, beta, el, eh)
    assert err == 0
    for r0 in range(0, spec.rows, 256):
        compare_grpo_rows(inp, f, dl, np.arange(r0, r0 + 256), old, ref, T, beta, el, eh, "fused pages")
    # same zero rows and (to within the idx element's summation order) the same gradient as fwd + bwd
    fs, dls, _ = run_gpu_grpo(inp, old, ref, T, beta, el, eh)
    assert torch.equal(f["is_clipped"], fs["is_clipped"])
    zf = (dl.reshape(spec.rows, -1).view(torch.int16) == 0).all(dim=1)
    zs = (dls.reshape(spec.rows, -1).view(torch.int16) == 0).all(dim=1)
    assert torch.equal(zf, zs) and int(zf.sum()) > spec.rows // 2
    diff = (dl.float() - dls.float()).abs()
    ulp = torch.maximum(dls.float().abs(), dl.float().abs()) * 2.0 ** -7
    assert bool((diff <= ulp + 1e-30).all())


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("V", [1, 9, 513, 4097, 40000, 65541, 151936])
@pytest.mark.parametrize("offset,extra", [(0, 0), (3, 1)])
@pytest.mark.parametrize("beta", [0.0, 0.05])
def test_fused_edge_shapes_every_row(dtype, V, offset, extra, beta):
    """Every row against the oracle twice: with dlogits rows out of phase with the logits
    (scalar-load variant), and with dlogits rows in the logits' own layout, where a long
    row's first 104 KB are held in shared memory between the sweeps and masked or zero rows
    are written by bulk stores; rows start at varying 16-byte phases when extra is odd.
    In place equals the same layout bit for bit."""
    B, L = 2, 5
    R = B * L
    seed = V * 7 + offset + int(beta * 100)
    x, idx, adv, mask, dloss = edge_inputs(B, L, V, dtype, offset, extra, seed)
    T, el, eh = f32(0.8), f32(0.2), f32(0.28)
    beta = f32(beta)
    xo = rows_f64(select_rows(x, np.arange(R)))
    lp, _ = oracle.selective_log_softmax(xo, idx.cpu().numpy(), T)
    g = torch.Generator().manual_seed(V)
    old = oracle.round_to_fp32(lp + torch.randn(R, generator=g).double().numpy() * 0.3)
    ref = oracle.round_to_fp32(lp + torch.randn(R, generator=g).double().numpy() * 0.1)
    inp = W.Inputs(W.get("tiny_fp32", B=B, L=L, V=V), x, idx, adv, mask, dloss, None, None, None, None)
    dl_buf = torch.empty(B * L * (V + 2) + 9, dtype=dtype, device=DEV)
    dl_view = torch.as_strided(dl_buf, (B, L, V), (L * (V + 2), V + 2, 1), 1 + offset)  # out of phase
    f, dl, err = run_gpu_fused(inp, old, ref, T, beta, el, eh, dlogits=dl_view)
    assert err == 0
    compare_grpo_rows(inp, f, dl, np.arange(R), old, ref, T, beta, el, eh, f"fused edge V={V}")
    x2, _ = strided_logits(B, L, V, dtype, offset, extra, seed)
    same_layout, _ = strided_logits(B, L, V, dtype, offset, extra, seed + 99)
    f_same, dl_same, err_same = run_gpu_fused(inp, old, ref, T, beta, el, eh, dlogits=same_layout)
    assert err_same == 0
    compare_grpo_rows(inp, f_same, dl_same, np.arange(R), old, ref, T, beta, el, eh, f"fused edge V={V} same phase")
    inp2 = W.Inputs(inp.spec, x2, idx, adv, mask, dloss, None, None, None, None)
    _, dl2, err2 = run_gpu_fused(inp2, old, ref, T, beta, el, eh, dlogits=x2)   # in place
    assert err2 == 0 and dl2.data_ptr() == x2.data_ptr()
    assert torch.equal(bf16_or_f32_bits(select_rows(dl2, np.arange(R))),
                       bf16_or_f32_bits(select_rows(dl_same, np.arange(R))))


@pytest.mark.parametrize("V", [65536, 100000, 151936, 158216])
@pytest.mark.parametrize("beta", [0.0, 0.05])
def test_fused_long_aligned_rows_every_row(V, beta):
    """Long bf16 rows with 16-byte aligned starts (the 512-thread fused kernel, which holds
    the first 104 KB of each row in shared memory and the rest in L2 between its two sweeps):
    every row against the oracle, including a row
    with -inf logits, a peaked row (p_idx near 1), masked and zero-advantage rows; in place
    equal bit for bit to out of place."""
    B, L = 2, 5
    R = B * L
    seed = V + int(beta * 100)
    x, idx, adv, mask, dloss = edge_inputs(B, L, V, torch.bfloat16, 0, 0, seed)
    x[0, 1, 7::977] = float("-inf")
    x[1, 2, int(idx[7])] += 30.0
    mask[3] = 0
    T, el, eh = f32(0.8), f32(0.2), f32(0.28)
    beta = f32(beta)
    xo = rows_f64(select_rows(x, np.arange(R)))
    lp, _ = oracle.selective_log_softmax(xo, idx.cpu().numpy(), T)
    g = torch.Generator().manual_seed(V)
    old = oracle.round_to_fp32(lp + torch.randn(R, generator=g).double().numpy() * 0.3)
    ref = oracle.round_to_fp32(lp + torch.randn(R, generator=g).double().numpy() * 0.1)
    inp = W.Inputs(W.get("tiny_fp32", B=B, L=L, V=V), x, idx, adv, mask, dloss, None, None, None, None)
    out = torch.empty(B, L, V, dtype=torch.bfloat16, device=DEV)
    f, dl, err = run_gpu_fused(inp, old, ref, T, beta, el, eh, dlogits=out)
    assert err == 0
    compare_grpo_rows(inp, f, dl, np.arange(R), old, ref, T, beta, el, eh, f"fused long rows V={V}")
    x2 = x.clone()
    inp2 = W.Inputs(inp.spec, x2, idx, adv, mask, dloss, None, None, None, None)
    f2, dl2, err2 = run_gpu_fused(inp2, old, ref, T, beta, el, eh, dlogits=x2)   # in place
    assert err2 == 0 and dl2.data_ptr() == x2.data_ptr()
    assert torch.equal(dl2.view(torch.int16), dl.view(torch.int16))
    for k in ("loss", "logp", "lse", "entropy"):
        assert torch.equal(f2[k], f[k]), k


def test_fused_long_rows_several_waves():
    """Several waves of rows at V = 151936 (800 rows, about 300 resident at once, so rows
    compete for L2 between their two sweeps): random masked rows and a run of 150 masked rows,
    a zero-advantage sequence with beta = 0 (zero rows decided after the statistic); every row
    against the oracle, in place equal bit for bit to out of place."""
    B, L, V = 8, 100, 151936
    R = B * L
    x, idx, adv, mask, dloss = edge_inputs(B, L, V, torch.bfloat16, 0, 0, 4242)
    mask[120:270] = 0
    adv[2] = 0.0
    T, beta, el, eh = f32(0.9), 0.0, f32(0.2), f32(0.28)
    xo = rows_f64(select_rows(x, np.arange(R)))
    lp, _ = oracle.selective_log_softmax(xo, idx.cpu().numpy(), T)
    del xo
    g = torch.Generator().manual_seed(17)
    old = oracle.round_to_fp32(lp + torch.randn(R, generator=g).double().numpy() * 0.3)
    inp = W.Inputs(W.get("tiny_fp32", B=B, L=L, V=V), x, idx, adv, mask, dloss, None, None, None, None)
    out = torch.empty(B, L, V, dtype=torch.bfloat16, device=DEV)
    f, dl, err = run_gpu_fused(inp, old, None, T, beta, el, eh, dlogits=out)
    assert err == 0
    for r0 in range(0, R, 50):
        compare_grpo_rows(inp, f, dl, np.arange(r0, r0 + 50), old, None, T, beta, el, eh, f"many rows {r0}")
    x2 = x.clone()
    inp2 = W.Inputs(inp.spec, x2, idx, adv, mask, dloss, None, None, None, None)
    f2, dl2, err2 = run_gpu_fused(inp2, old, None, T, beta, el, eh, dlogits=x2)
    assert err2 == 0
    assert torch.equal(dl2.view(torch.int16), dl.view(torch.int16))
    assert torch.equal(f2["logp"], f["logp"]) and torch.equal(f2["entropy"], f["entropy"])


# ---------------------------------------------------------------------------
# entropy backward
# ---------------------------------------------------------------------------

def check_entropy_grad(dl_gpu, x_orc, up, T, H_gpu, lse_gpu, what):
    """GPU entropy gradient rows vs the oracle.  Each element is g p_j (log p_j + H); the
    forward's fp32 lse and H enter it, so besides 1 bf16 ulp (or 1e-5 relative for fp32)
    an element may differ by |g| p_j (|dlse| (|log p_j + H| + 1) + |dH|
    + 4e-7 (|log p_j| + |H| + 1) (1 + |log p_j + H|)), with dlse, dH the forward's actual
    deviations from the oracle on that row."""
    odl, g = oracle.entropy_from_logits_bwd(x_orc, up, T)
    z, lse = oracle.log_softmax_rows(x_orc, T)
    H = oracle.entropy_from_logits(x_orc, T)
    with np.errstate(all="ignore"):
        logp = z - lse[:, None]
        p = np.exp(logp)
        w = np.abs(logp + H[:, None])
        dlse = np.abs(np.asarray(lse_gpu, dtype=np.float64) - lse)[:, None]
        dH = np.abs(np.asarray(H_gpu, dtype=np.float64) - H)[:, None]
        bound = np.abs(g)[:, None] * p * (dlse * (w + 1) + dH + 4e-7 * (np.abs(logp) + np.abs(H)[:, None] + 1) * (1 + w))
        bound = np.nan_to_num(bound, nan=0.0, posinf=0.0)
    zero = g == 0.0
    if np.any(zero):
        assert_plus_zero(dl_gpu[torch.from_numpy(np.nonzero(zero)[0]).to(dl_gpu.device)], f"{what} zero rows")
    live = np.nonzero(~zero)[0]
    if len(live) == 0:
        return
    sub = rows_f64(dl_gpu[torch.from_numpy(live).to(dl_gpu.device)])
    o, bd = odl[live], bound[live]
    if dl_gpu.dtype == torch.bfloat16:
        ob = oracle.bf16_bits_to_fp64(oracle.round_to_bf16_bits(o))
        ulp = np.where(np.abs(ob) >= 2.0 ** -126, np.ldexp(1.0, np.frexp(np.abs(ob))[1] - 8), 2.0 ** -133)
        tol = ulp + bd + np.where(np.abs(o) < 2.0 ** -126, 2.0 ** -126, 0.0)
    else:
        tol = 1e-5 * np.abs(o) + bd + np.where(np.abs(o) < 2.0 ** -126, 2.0 ** -126, 0.0)
    err = np.abs(sub - o)
    assert np.array_equal(np.isnan(sub), np.isnan(o)), f"{what}: NaN pattern differs"
    bad = (err > tol) & ~np.isnan(o)
    assert not np.any(bad), f"{what}: {int(bad.sum())} elements out of tolerance, worst {err[bad].max():.3g}"
    assert np.all(np.abs(np.nansum(sub, axis=1)) <= np.abs(g[live]) * (1e-3 + sub.shape[1] * 2.0 ** -8))


@pytest.mark.parametrize("seed", [0, 1])
def test_entropy_bwd_tiny_every_row(seed):
    spec = W.get("tiny_fp32")
    inp = W.generate(spec, seed, device=DEV)
    T = 0.8
    H, lse = rp.entropy_from_logits(inp.logits, T=T, return_lse=True)
    up = torch.randn(spec.rows, generator=torch.Generator().manual_seed(seed)).float()
    up[1] = 0.0
    up[4] = -0.0
    dl = rp.entropy_from_logits_bwd(inp.logits, up.to(DEV), lse, H, T=T)
    torch.cuda.synchronize()
    x = rows_f64(inp.logits.reshape(-1, spec.V))
    assert_scalar_close(lse, oracle.log_softmax_rows(x, T)[1], "entropy lse output")
    check_entropy_grad(dl.reshape(spec.rows, -1), x, up.double().numpy(), T, H.cpu().numpy(), lse.cpu().numpy(),
                       "entropy bwd tiny")


def test_entropy_bwd_v32000_sampled_rows_with_peaks():
    """(16, 4096, 32000) bf16 at full size, as the benchmark's entropy-backward step runs it."""
    spec = W.get("entropy_slsm_b16_l4096_v32000")
    inp = W.generate(spec, 2, device=DEV)
    T = 1.0
    H, lse = rp.entropy_from_logits(inp.logits, T=T, return_lse=True)
    up = torch.full((spec.rows,), 1.0 / spec.rows, device=DEV)
    dl = rp.entropy_from_logits_bwd(inp.logits, up, lse, H, T=T)
    torch.cuda.synchronize()
    peaked = torch.nonzero(inp.logits.float().amax(dim=-1).reshape(-1) > 14.0)[:, 0].cpu().numpy()
    rows = np.unique(np.concatenate([W.sample_rows(spec.rows, 24, 4), peaked[:16]]))
    x = rows_f64(select_rows(inp.logits, rows))
    r_t = torch.from_numpy(rows).to(DEV)
    check_entropy_grad(select_rows(dl, rows), x, np.full(len(rows), 1.0 / spec.rows), T,
                       H[r_t].cpu().numpy(), lse[r_t].cpu().numpy(), "entropy bwd v32000")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("V", [1, 9, 513, 4097, 40000])
@pytest.mark.parametrize("offset,extra", [(0, 0), (3, 1)])
def test_entropy_bwd_edge_shapes_every_row(dtype, V, offset, extra):
    B, L = 2, 5
    R = B * L
    seed = V * 11 + offset
    x, _ = strided_logits(B, L, V, dtype, offset, extra, seed)
    if V > 4:
        x[0, 1, 3] = float("-inf")        # a masked-out vocabulary entry: p = 0, adds 0
    T = 1.3
    H, lse = rp.entropy_from_logits(x, T=T, return_lse=True)
    up = torch.randn(R, generator=torch.Generator().manual_seed(seed)).float()
    up[2] = 0.0
    dl_buf = torch.empty(B * L * (V + 2) + 9, dtype=dtype, device=DEV)
    dl_view = torch.as_strided(dl_buf, (B, L, V), (L * (V + 2), V + 2, 1), 1 + offset)  # out of phase
    dl = rp.entropy_from_logits_bwd(x, up.to(DEV), lse, H, T=T, dlogits=dl_view)
    torch.cuda.synchronize()
    xo = rows_f64(select_rows(x, np.arange(R)))
    check_entropy_grad(select_rows(dl, np.arange(R)), xo, up.double().numpy(), T, H.cpu().numpy(),
                       lse.cpu().numpy(), f"entropy bwd edge V={V}")
    x2, _ = strided_logits(B, L, V, dtype, offset, extra, seed)
    if V > 4:
        x2[0, 1, 3] = float("-inf")
    same, _ = strided_logits(B, L, V, dtype, offset, extra, seed + 5)
    d_same = rp.entropy_from_logits_bwd(x2, up.to(DEV), lse, H, T=T, dlogits=same)
    d_in = rp.entropy_from_logits_bwd(x2, up.to(DEV), lse, H, T=T, dlogits=x2)
    torch.cuda.synchronize()
    assert torch.equal(bf16_or_f32_bits(select_rows(d_in, np.arange(R))),
                       bf16_or_f32_bits(select_rows(d_same, np.arange(R))))


# ---------------------------------------------------------------------------
# sequence-level GRPO: slsm fwd -> grpo_seq_terms -> slsm bwd
# ---------------------------------------------------------------------------

def run_seq_pipeline(inp, old, ref, T, beta, el, eh):
    spec = inp.spec
    t = lambda a: None if a is None else torch.as_tensor(a, dtype=torch.float32).to(DEV)
    logp, lse = rp.selective_log_softmax_fwd(inp.logits, inp.idx, T=T)
    st = rp.grpo_seq_terms(logp, inp.adv, inp.dloss, B=spec.B, L=spec.L, beta=beta, eps_low=el, eps_high=eh,
                           old_logp=t(old), ref_logp=t(ref), mask=inp.mask)
    dl = rp.selective_log_softmax_bwd(inp.logits, inp.idx, st["dlogp"], lse, T=T)
    torch.cuda.synchronize()
    return logp, lse, st, dl


def compare_seq(inp, old, ref, T, beta, el, eh, logp, lse, st, dl, tag, rows=None, seqs=None):
    """The terms of the sequences `seqs` (default: every sequence) and the dlogits of `rows`
    (default: every row of those sequences) against the oracle.  The per-sequence ratio
    depends on the forward's fp32 logp of all the sequence's tokens, so the budget of each
    term includes |A| s max|dlogp| (and the KL's own dependence)."""
    spec = inp.spec
    B, L = spec.B, spec.L
    seqs = np.arange(B) if seqs is None else np.sort(np.asarray(seqs))
    Bs = len(seqs)
    srows = (seqs[:, None] * L + np.arange(L)[None, :]).reshape(-1)     # rows of the checked sequences
    idx_all = inp.idx.cpu().numpy()
    idx = idx_all[srows]
    mask = None if inp.mask is None else inp.mask.cpu().numpy()[srows]
    dloss = inp.dloss.cpu().numpy().astype(np.float64)[srows]
    A = inp.adv.cpu().numpy().astype(np.float64)[seqs]
    o_old = None if old is None else np.asarray(old, dtype=np.float64)[srows]
    o_ref = None if ref is None else np.asarray(ref, dtype=np.float64)[srows]
    lp_o = oracle_logp(inp.logits, idx_all, T, rows=srows)
    terms = oracle.grpo_seq_terms(lp_o, o_old, o_ref, A, mask, dloss, Bs, L, beta, el, eh)
    dlp = np.abs(logp.double().cpu().numpy()[srows] - lp_o)
    m = np.ones((Bs, L), bool) if mask is None else mask.reshape(Bs, L) != 0
    dmax = np.where(m, dlp.reshape(Bs, L), 0.0).max(axis=1)                      # per sequence
    s = terms["seq_ratio"]
    assert_scalar_close(st["seq_ratio"].cpu()[seqs], s, f"{tag} seq ratio", atol=0.0,
                        rtol=1e-5 + float(np.max(dmax) * 1.01))
    lo, hi = 1 - el, 1 + eh
    amb_seq = (A != 0) & ((np.abs(s - lo) <= 1e-5 * lo) | (np.abs(s - hi) <= 1e-5 * hi))
    assert np.array_equal(st["seq_is_clipped"].cpu().numpy().astype(bool)[seqs][~amb_seq],
                          terms["seq_is_clipped"][~amb_seq])
    W = np.where(m, dloss.reshape(Bs, L), 0.0).sum(axis=1)
    n = np.maximum(m.sum(axis=1), 1)
    pg_sens = (np.abs(A) * s)[:, None] * dmax[:, None]                             # |d pg| bound
    kl_sens = (beta * np.exp(np.asarray(o_ref).reshape(Bs, L) - lp_o.reshape(Bs, L)) * dlp.reshape(Bs, L)
               if (beta != 0 and o_ref is not None) else np.zeros((Bs, L)))
    loss_budget = (pg_sens + kl_sens).reshape(-1) * 1.01
    assert_scalar_close(st["loss"].cpu()[srows], terms["loss"], f"{tag} loss", atol=1e-5 + float(loss_budget.max()))
    dlogp_budget = ((W * np.abs(A) * s / n * 2 * dmax)[:, None] + kl_sens * np.abs(dloss.reshape(Bs, L))).reshape(-1)
    got = st["dlogp"].double().cpu().numpy()[srows]
    err = np.abs(got - terms["dlogp"])
    assert np.all(err <= 1e-5 * np.abs(terms["dlogp"]) + 1e-7 * np.abs(W).max() + dlogp_budget * 1.01), \
        f"{tag} dlogp: worst {err.max():.3g}"
    # dlogits: the row factor is dlogp / T with the GPU's own dlogp; its deviation is the budget
    rows = srows if rows is None else np.asarray(rows)
    pos = np.searchsorted(srows, rows)
    assert np.array_equal(srows[pos], rows), "rows outside the checked sequences"
    x = rows_f64(select_rows(inp.logits, rows))
    odl = oracle.softmax_gather_grad(x, idx[pos], terms["dlogp"][pos] / T, T)
    g = terms["dlogp"][pos] / T
    with np.errstate(divide="ignore", invalid="ignore"):
        rho = np.where(g != 0, err[pos] / np.abs(terms["dlogp"][pos]), 0.0)
    rho = rho + np.abs(lse.double().cpu().numpy()[rows] - oracle.selective_log_softmax(x, idx[pos], T)[1]) + 1e-6
    amb = (rho > 2.0 ** -10) | np.repeat(amb_seq, L)[pos]
    assert amb.sum() <= max(2, 0.01 * len(rows)), f"{tag}: {amb.sum()} ambiguous rows"
    assert_grad_rows(select_rows(dl, rows), odl, g, amb, f"{tag} dlogits", rho=rho)


@pytest.mark.parametrize("seed", [0, 1])
def test_seq_level_tiny_every_row(seed):
    spec = W.get("tiny_fp32", L=16)
    inp = W.generate(spec, seed, device=DEV)
    T, beta, el, eh = f32(spec.T), f32(spec.beta), f32(spec.eps_low), f32(spec.eps_high)
    lp = oracle_logp(inp.logits, inp.idx.cpu().numpy(), T)
    old, ref = near_logp_inputs(inp, lp)
    out = run_seq_pipeline(inp, old, ref, T, beta, el, eh)
    compare_seq(inp, old, ref, T, beta, el, eh, *out, f"seq tiny s{seed}")


def test_seq_level_pages_shape_every_row():
    """B=4, L=512, V=32000 bf16 with a completion mask; beta = 0: zero-advantage and clipped
    sequences give +0.0 rows for all their tokens."""
    spec = W.get("grpo_b4_l512_v32000", old_sigma=0.02)
    inp = W.generate(spec, 3, device=DEV)
    T, beta, el, eh = f32(spec.T), 0.0, f32(spec.eps_low), f32(spec.eps_high)
    lp = oracle_logp(inp.logits, inp.idx.cpu().numpy(), T)
    old, ref = near_logp_inputs(inp, lp)
    logp, lse, st, dl = run_seq_pipeline(inp, old, ref, T, beta, el, eh)
    for r0 in range(0, spec.rows, 512):
        compare_seq(inp, old, ref, T, beta, el, eh, logp, lse, st, dl, "seq pages", rows=np.arange(r0, r0 + 512))
    zero_seq = torch.nonzero(inp.adv == 0)[:, 0]
    assert len(zero_seq) == 2
    assert_plus_zero(dl[zero_seq], "zero-advantage sequences")


def test_seq_level_beta_and_all_masked_sequence():
    spec = W.get("grpo_qwen3_b16_l1024_v151936", B=4, L=64, V=1000, group_size=4)
    inp = W.generate(spec, 4, device=DEV)
    inp.mask.view(4, 64)[2] = 0                      # a sequence with no tokens: ratio 1, zero terms
    inp.dloss.view(4, 64)[2] = 0.0
    T, beta, el, eh = f32(spec.T), f32(spec.beta), f32(spec.eps_low), f32(spec.eps_high)
    lp = oracle_logp(inp.logits, inp.idx.cpu().numpy(), T)
    old, ref = near_logp_inputs(inp, lp)
    out = run_seq_pipeline(inp, old, ref, T, beta, el, eh)
    compare_seq(inp, old, ref, T, beta, el, eh, *out, "seq beta")
    assert float(out[2]["seq_ratio"][2]) == 1.0
    assert_plus_zero(out[3][2], "all-masked sequence")


def test_seq_level_qwen3_full_size_sampled():
    """(16, 1024, 151936) bf16, beta = 0.04, in the launch configuration the benchmark's
    sequence-level step times.  Three whole sequences go through the oracle (their ratio
    sums over all their tokens) with 48 of their rows checked element by element; every
    row is checked for masked rows being +0.0 and for a row sum of ~0."""
    spec = W.get("grpo_qwen3_b16_l1024_v151936")
    inp = W.generate(spec, 1, device=DEV)
    T, beta, el, eh = f32(spec.T), f32(spec.beta), f32(spec.eps_low), f32(spec.eps_high)
    seqs = np.array([0, 7, 15])
    srows = (seqs[:, None] * spec.L + np.arange(spec.L)[None, :]).reshape(-1)
    lp_all = torch_logp(inp.logits, inp.idx, T).double().cpu().numpy()
    lp_all[srows] = oracle_logp(inp.logits, inp.idx.cpu().numpy(), T, rows=srows)
    old, ref = near_logp_inputs(inp, lp_all)
    logp, lse, st, dl = run_seq_pipeline(inp, old, ref, T, beta, el, eh)
    live = inp.mask.cpu().numpy()[srows] != 0
    rows = np.unique(np.concatenate([srows[live][W.sample_rows(int(live.sum()), 40, 6)],
                                     srows[~live][:8]]))
    compare_seq(inp, old, ref, T, beta, el, eh, logp, lse, st, dl, "seq qwen3", rows=rows, seqs=seqs)
    masked = inp.mask == 0
    assert bool(masked.any())
    assert_plus_zero(dl.reshape(-1, spec.V)[masked], "masked dlogits rows")
    g = st["dlogp"].abs() / T
    rs = dl.float().sum(dim=-1).reshape(-1).abs()
    assert bool(torch.all(rs <= g * (1e-3 + spec.V * 2.0 ** -8)))


@pytest.mark.parametrize("L", [1, 31, 256, 257, 700, 1024, 1025, 3000])
def test_seq_terms_every_length_against_oracle(L):
    """grpo_seq_terms alone on fp32 inputs, across the register-resident kernels (L <= 256,
    512, 1024) and the two-pass one (L > 1024): a masked tail, a fully masked sequence, one
    with A = 0, and beta on."""
    B = 5
    g = torch.Generator().manual_seed(L)
    logp = -torch.rand(B * L, generator=g).float() * 4
    old = (logp + torch.randn(B * L, generator=g) * 0.05).float()
    ref = (logp + torch.randn(B * L, generator=g) * 0.05).float()
    mask = (torch.rand(B * L, generator=g) > 0.15).to(torch.uint8)
    mask.view(B, L)[1] = 0
    dloss = (torch.rand(B * L, generator=g) / L).float() * mask.float()
    adv = torch.randn(B, generator=g).float()
    adv[2] = 0.0
    beta, el, eh = 0.04, 0.2, 0.28
    st = rp.grpo_seq_terms(logp.to(DEV), adv.to(DEV), dloss.to(DEV), B=B, L=L, beta=beta, eps_low=el, eps_high=eh,
                           old_logp=old.to(DEV), ref_logp=ref.to(DEV), mask=mask.to(DEV))
    torch.cuda.synchronize()
    t = oracle.grpo_seq_terms(logp.double().numpy(), old.double().numpy(), ref.double().numpy(),
                              adv.double().numpy(), mask.numpy(), dloss.double().numpy(), B, L, beta, el, eh)
    assert_scalar_close(st["seq_ratio"], t["seq_ratio"], f"L={L} seq ratio")
    lo, hi = 1 - el, 1 + eh
    s = t["seq_ratio"]
    amb = (np.abs(s - lo) <= 1e-5 * lo) | (np.abs(s - hi) <= 1e-5 * hi)
    assert np.array_equal(st["seq_is_clipped"].cpu().numpy().astype(bool)[~amb], t["seq_is_clipped"][~amb])
    assert_scalar_close(st["loss"], t["loss"], f"L={L} loss")
    assert_scalar_close(st["kl"], t["kl"], f"L={L} kl")
    W = np.abs(dloss.double().numpy()).reshape(B, L).sum(axis=1)
    got = st["dlogp"].double().cpu().numpy()
    err = np.abs(got - t["dlogp"])
    assert np.all(err <= 1e-5 * np.abs(t["dlogp"]) + 1e-6 * np.repeat(W * np.abs(adv.numpy()) + beta, L)), \
        f"L={L} dlogp: worst {err.max():.3g}"
    masked = mask.numpy() == 0
    for k in ("loss", "kl", "dlogp"):
        v = st[k].cpu().numpy()[masked]
        assert np.all(v == 0.0) and not np.any(np.signbit(v)), f"L={L} masked {k} must be +0.0"
    assert float(st["seq_ratio"][1]) == 1.0


# ---------------------------------------------------------------------------
# size limits: a million-entry vocabulary row, sixteen million rows
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_vocabulary_of_a_million_every_element(dtype):
    """V = 2^20 + 3 (a scalar tail after the last 16-byte vector): four rows with idx at the
    first column, the last column and two inside, every output and every dlogits element
    against the oracle.  Each thread's partial sums cover ~4096 terms here, 15 times more
    than at V = 151936; the scalar tolerances are unchanged."""
    spec = W.get("tiny_fp32", B=1, L=4, V=(1 << 20) + 3, dtype=dtype, adv="plus_minus_one")
    inp = W.generate(spec, 5, device=DEV)
    inp.idx[0] = 0
    inp.idx[1] = spec.V - 1
    T, beta, el, eh = f32(0.8), f32(0.04), f32(spec.eps_low), f32(spec.eps_high)
    lp = oracle_logp(inp.logits, inp.idx.cpu().numpy(), T)
    old, ref = near_logp_inputs(inp, lp)
    f, dl, err = run_gpu_grpo(inp, old, ref, T, beta, el, eh)
    assert err == 0
    compare_grpo_rows(inp, f, dl, np.arange(spec.rows), old, ref, T, beta, el, eh, f"V=2^20+3 {dtype}")


def test_sixteen_million_rows_sampled():
    """B = L = 4096 (16,777,216 rows, one CTA each) with V = 8: 4096 sampled rows against the
    oracle, and over every row: masked rows and zero-advantage sequences (beta = 0) give
    +0.0 gradient rows, the others sum to ~0."""
    spec = W.get("grpo_b4_l512_v32000", B=4096, L=4096, V=8)
    inp = W.generate(spec, 7, device=DEV, rows_per_chunk=1 << 20)
    T, beta, el, eh = f32(spec.T), 0.0, f32(spec.eps_low), f32(spec.eps_high)
    rows = W.sample_rows(spec.rows, 4096, 9)
    lp_all = torch_logp(inp.logits, inp.idx, T, chunk=1 << 20).double().cpu().numpy()
    lp_all[rows] = oracle.selective_log_softmax(rows_f64(select_rows(inp.logits, rows)),
                                                inp.idx.cpu().numpy()[rows], T)[0]
    old, ref = near_logp_inputs(inp, lp_all)
    f, dl, err = run_gpu_grpo(inp, old, ref, T, beta, el, eh)
    assert err == 0
    compare_grpo_rows(inp, f, dl, rows, old, ref, T, beta, el, eh, "16M rows")
    flat = dl.reshape(-1, spec.V)
    zero_rows = (inp.mask == 0) | (inp.adv.repeat_interleave(spec.L) == 0)
    assert bool(zero_rows.any()) and bool((~zero_rows).any())
    assert_plus_zero(flat[zero_rows], "masked and zero-advantage rows")
    rs = flat.float().sum(dim=-1).abs()
    bound = flat.float().abs().sum(dim=-1) * 2.0 ** -8 + 1e-30
    assert bool(torch.all(rs <= bound)), "row sums"
