"""grpo_fused_linear_noalloc, the variant of grpo_fused_linear for callers that cannot
allocate device memory when the loss runs: its scratch is a fixed array inside the
library, so the caller passes only inputs and outputs.  Checked through the C ABI against
grpo_fused_linear (which takes a workspace from the caller) on two calls in a row, with
different inputs, so that the second call also shows that what the first left in the
shared array does not leak into its results.  This file is collected last on purpose.
"""

import numpy as np
import pytest
import torch

import oracle
from parity_util import assert_scalar_close, rows_f64
from rl_fine_tuning_pass_gb300 import binding as rp

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]
DEV = "cuda"


@pytest.fixture(scope="module")
def lib():
    from rl_fine_tuning_pass_gb300.build import build
    build()
    return rp.load_library()


def inputs(seed, B=2, L=21, H=64, V=1003, T=0.9):
    """Seeded inputs; old / ref sit near the oracle's logp of h W^T (old within about 0.3,
    ref 0.1), so that rows fall on both sides of the clip range and the KL term is live."""
    g = torch.Generator().manual_seed(seed)
    R = B * L
    h = torch.randn(R, H, generator=g).to(torch.bfloat16)
    W = (torch.randn(V, H, generator=g) * (2.0 / np.sqrt(H))).to(torch.bfloat16)
    idx = torch.randint(0, V, (R,), generator=g)
    adv = torch.randn(B, generator=g).float()
    mask = (torch.rand(R, generator=g) > 0.2).to(torch.uint8)
    dloss = (torch.rand(R, generator=g) + 0.1).float() * mask.float()
    lp, _ = oracle.selective_log_softmax(rows_f64(h) @ rows_f64(W).T, idx.numpy(), T)
    old = torch.from_numpy(oracle.round_to_fp32(lp + 0.3 * torch.randn(R, generator=g).double().numpy())).float()
    ref = torch.from_numpy(oracle.round_to_fp32(lp + 0.1 * torch.randn(R, generator=g).double().numpy())).float()
    d = lambda t: t.to(DEV)
    return dict(h=d(h), W=d(W), idx=d(idx), adv=d(adv), mask=d(mask), dloss=d(dloss), old=d(old), ref=d(ref),
                B=B, L=L, H=H, V=V, T=T, beta=0.04, el=0.2, eh=0.28)


def call_noalloc(lib, x, chunk):
    R, H, V = x["B"] * x["L"], x["H"], x["V"]
    f32 = dict(dtype=torch.float32, device=DEV)
    out = {"loss": torch.empty(R, **f32), "logp": torch.empty(R, **f32), "lse": torch.empty(R, **f32),
           "kl": torch.empty(R, **f32), "is_clipped": torch.empty(R, dtype=torch.uint8, device=DEV),
           "entropy": torch.empty(R, **f32), "grad_hidden": torch.empty(R, H, **f32),
           "grad_weight": torch.zeros(V, H, **f32)}
    st = lib.grpo_fused_linear_noalloc(
        x["h"].data_ptr(), x["W"].data_ptr(), x["B"], x["L"], H, V, x["idx"].data_ptr(), x["old"].data_ptr(),
        x["ref"].data_ptr(), x["adv"].data_ptr(), x["mask"].data_ptr(), x["dloss"].data_ptr(), x["T"], x["beta"],
        x["el"], x["eh"], chunk, out["loss"].data_ptr(), out["logp"].data_ptr(), out["lse"].data_ptr(),
        out["kl"].data_ptr(), out["is_clipped"].data_ptr(), out["entropy"].data_ptr(), out["grad_hidden"].data_ptr(),
        out["grad_weight"].data_ptr(), None, torch.cuda.current_stream().cuda_stream)
    return st, out


def call_with_workspace(x, chunk):
    return rp.grpo_fused_linear(x["h"], x["W"], x["idx"], x["adv"], x["dloss"], B=x["B"], L=x["L"], T=x["T"],
                                beta=x["beta"], eps_low=x["el"], eps_high=x["eh"], old_logp=x["old"],
                                ref_logp=x["ref"], mask=x["mask"], chunk_rows=chunk)


def gradient_bounds(x):
    """The parity tests' gradient tolerance (2^-8 of |dlogits| |W| and |dlogits|^T |h|, for
    the bf16 rounding of dlogits, plus 1e-5 relative), from the oracle's dlogits; doubled,
    since both entry points are compared, each within it of the oracle."""
    hf, Wf = rows_f64(x["h"]), rows_f64(x["W"])
    adv = oracle.per_row(x["adv"].cpu().numpy(), x["L"])
    g = lambda t: t.double().cpu().numpy()
    _, gh, gW, dx = oracle.fused_linear_grpo(hf, Wf, x["idx"].cpu().numpy(), g(x["old"]), g(x["ref"]), adv,
                                             x["mask"].cpu().numpy(), g(x["dloss"]), x["T"], x["beta"], x["el"],
                                             x["eh"])
    bh = 2 * (2.0 ** -8 * (np.abs(dx) @ np.abs(Wf)) + 1e-5 * np.abs(gh)) + 1e-7
    bW = 2 * (2.0 ** -8 * (np.abs(dx).T @ np.abs(hf)) + 1e-5 * np.abs(gW)) + 1e-7
    return bh, bW


def test_noalloc_matches_the_workspace_entry_point_on_two_calls(lib):
    for seed in (1, 2):
        x = inputs(seed)
        st, got = call_noalloc(lib, x, 16)
        assert st == rp.GRPO_OK, rp.status_string(st)
        want = call_with_workspace(x, 16)
        torch.cuda.synchronize()
        # the same kernels; grad_hidden's K splits may be fewer in the fixed array, which
        # changes only its fp32 summation order: the parity tests' tolerances
        for k in ("loss", "logp", "lse", "kl", "entropy"):
            assert_scalar_close(got[k], want[k].double().cpu().numpy(), f"call {seed}: {k}")
        assert torch.equal(got["is_clipped"], want["is_clipped"]), f"call {seed}: is_clipped"
        bh, bW = gradient_bounds(x)
        for k, bound in (("grad_hidden", bh), ("grad_weight", bW)):
            diff = (got[k] - want[k]).abs().double().cpu().numpy()
            assert np.all(diff <= bound), f"call {seed}: {k}, worst {diff.max():.3g}"


def compare_to_workspace_entry_point(lib, x, chunk, what):
    st, got = call_noalloc(lib, x, chunk)
    assert st == rp.GRPO_OK, rp.status_string(st)
    want = call_with_workspace(x, chunk)
    torch.cuda.synchronize()
    for k in ("loss", "logp", "lse", "kl", "entropy"):
        assert_scalar_close(got[k], want[k].double().cpu().numpy(), f"{what}: {k}")
    assert torch.equal(got["is_clipped"], want["is_clipped"]), f"{what}: is_clipped"
    bh, bW = gradient_bounds(x)
    for k, bound in (("grad_hidden", bh), ("grad_weight", bW)):
        diff = (got[k] - want[k]).abs().double().cpu().numpy()
        assert np.all(diff <= bound), f"{what}: {k}, worst {diff.max():.3g}"


@pytest.mark.parametrize("V", [151936, 151935])
def test_noalloc_at_the_limit_of_its_array(lib, V):
    """The largest chunk that fits the fixed array at the Qwen3 vocabulary (with H = 64: 103
    rows; the chunk buffers and one split of grad_hidden then fill 33.30 of its 33.55 MB, and
    104 rows would need 33.62), with V a multiple of 8 and not: rejected one row above it, and
    equal to grpo_fused_linear at it."""
    x = inputs(3, V=V, H=64, B=1, L=110)
    st, _ = call_noalloc(lib, x, 104)
    assert st == rp.GRPO_ERR_UNSUPPORTED
    compare_to_workspace_entry_point(lib, x, 103, f"V={V} chunk 103")
