"""The row-pass entry points inside a CUDA graph: a GRPO forward + backward step captured
once and replayed gives the eager results bit for bit (the kernels are launched with
programmatic stream serialization, which capture turns into programmatic graph edges)."""

import pytest
import torch

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


def step(inp, old, ref, spec, dlogits, out):
    f = rp.grpo_loss_fwd(inp.logits, inp.idx, inp.adv, T=spec.T, beta=spec.beta, eps_low=spec.eps_low,
                         eps_high=spec.eps_high, old_logp=old, ref_logp=ref, mask=inp.mask, with_entropy=True)
    rp.grpo_loss_bwd(inp.logits, inp.idx, inp.adv, inp.dloss, f["logp"], f["lse"], T=spec.T, beta=spec.beta,
                     eps_low=spec.eps_low, eps_high=spec.eps_high, old_logp=old, ref_logp=ref, mask=inp.mask,
                     dlogits=dlogits)
    for k in ("loss", "logp", "lse", "entropy"):
        out[k].copy_(f[k])


@pytest.mark.parametrize("name", ["tiny_fp32", "grpo_b4_l512_v32000"])
def test_grpo_step_replays_in_a_cuda_graph(name):
    spec = W.get(name)
    inp = W.generate(spec, 0, device=DEV)
    logp0, _ = rp.selective_log_softmax_fwd(inp.logits, inp.idx, T=spec.T)
    old = (logp0 + inp.old_offset).contiguous() if inp.old_offset is not None else None
    ref = (logp0 + inp.ref_offset).contiguous() if (inp.ref_offset is not None and spec.beta) else None
    R = spec.rows
    eager = {k: torch.empty(R, device=DEV) for k in ("loss", "logp", "lse", "entropy")}
    dl_eager = torch.empty_like(inp.logits)
    step(inp, old, ref, spec, dl_eager, eager)

    graphed = {k: torch.empty(R, device=DEV) for k in ("loss", "logp", "lse", "entropy")}
    dl_graph = torch.empty_like(inp.logits)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):                      # warm up on the side stream, as capture wants
        step(inp, old, ref, spec, dl_graph, graphed)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(inp, old, ref, spec, dl_graph, graphed)
    dl_graph.zero_()
    for v in graphed.values():
        v.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for k in eager:
        assert torch.equal(eager[k], graphed[k]), k
    assert torch.equal(dl_eager.view(torch.uint8), dl_graph.view(torch.uint8))


def test_fused_linear_replays_in_a_cuda_graph_and_follows_the_mask():
    """grpo_fused_linear in a CUDA graph: the rows of each chunk are picked on the device, so
    the captured call needs no host synchronisation, and a replay after the mask has changed
    (in place) packs the new unmasked rows.  Each replay equals an eager call on the same
    inputs bit for bit (grad_weight accumulated from zero)."""
    g = torch.Generator().manual_seed(7)
    B, L, H, V, chunk = 3, 40, 64, 1003, 32
    R = B * L
    h = torch.randn(R, H, generator=g).to(torch.bfloat16).to(DEV)
    Wt = (torch.randn(V, H, generator=g) * 0.25).to(torch.bfloat16).to(DEV)
    idx = torch.randint(0, V, (R,), generator=g).to(DEV)
    adv = torch.randn(B, generator=g).float().to(DEV)
    mask = (torch.rand(R, generator=g) > 0.3).to(torch.uint8).to(DEV)
    dloss = (torch.rand(R, generator=g) + 0.1).float().to(DEV)
    ws = torch.empty(rp.grpo_fused_linear_workspace_size(H, V, chunk), dtype=torch.uint8, device=DEV)
    kw = dict(B=B, L=L, T=0.9, beta=0.0, eps_low=0.2, eps_high=0.28, mask=mask, chunk_rows=chunk, workspace=ws)

    def eager():
        gw = torch.zeros(V, H, device=DEV)
        out = rp.grpo_fused_linear(h, Wt, idx, adv, dloss, grad_weight=gw, **kw)
        torch.cuda.synchronize()
        return {k: v.clone() for k, v in out.items()}

    gw = torch.zeros(V, H, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):                      # warm up (set-up of the GEMM launches) on the side stream
        rp.grpo_fused_linear(h, Wt, idx, adv, dloss, grad_weight=gw, **kw)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        captured = rp.grpo_fused_linear(h, Wt, idx, adv, dloss, grad_weight=gw, **kw)
    for new_mask in (None, (torch.arange(R, device=DEV) % 7 != 3).to(torch.uint8)):
        if new_mask is not None:
            mask.copy_(new_mask)
        want = eager()
        gw.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for k in ("loss", "logp", "lse", "kl", "is_clipped", "entropy", "grad_hidden", "grad_weight"):
            assert torch.equal(captured[k], want[k]), k
