"""bench.py's end-to-end path on the GPU: the batch cut into parts of whole sequences, with
host->device copies, kernels and device->host copies on three streams, must return exactly
what the device-resident step computes on the whole batch (same kernels and launch shapes;
rows are independent)."""
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from rl_fine_tuning_pass_gb300 import binding as rp  # noqa: E402
from rl_fine_tuning_pass_gb300 import workloads as W  # noqa: E402

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _library():
    from rl_fine_tuning_pass_gb300.build import build
    build()
    rp.load_library()


def _device_outputs(step):
    for _, fn in step.kernels:
        fn()
    torch.cuda.synchronize()
    out = {"dlogits": step.dlogits.detach().cpu().clone()}
    if isinstance(step, bench.SeqStep):
        out["loss"] = step.out["loss"].cpu().clone()
    elif isinstance(step, bench.EntropyBwdStep):
        out["entropy"] = step.H.cpu().clone()
    elif isinstance(step, bench.EntropySlsmStep):
        out.update(entropy=step.H.cpu().clone(), logp=step.logp.cpu().clone(), lse=step.lse.cpu().clone())
    else:
        out["loss"] = step.out["loss"].cpu().clone()
    return out


@pytest.mark.parametrize("case", ["grpo", "grpo_token_ranges", "fused", "seq", "vocab2", "slsm", "entropy_bwd"])
def test_pipelined_e2e_matches_device_step(case):
    if case in ("slsm", "entropy_bwd"):
        spec = W.get("entropy_slsm_b16_l4096_v32000", L=128)
    else:
        spec = W.get("grpo_b4_l512_v32000")
    step = bench.make_step(spec, 0, "cuda", fused=case == "fused", vocab_shards=2 if case == "vocab2" else 0,
                           seq_level=case == "seq", entropy_bwd=case == "entropy_bwd")
    want = _device_outputs(step)
    if case == "grpo_token_ranges":          # 16 parts: each sequence in four token ranges
        step.E2E_PART_BYTES = 8 << 20
    step.e2e_setup()
    if case == "grpo_token_ranges":
        assert len(step.e2e_bounds) == 16 and all(b1 - b0 == 1 for b0, b1, _, _ in step.e2e_bounds)
    assert len(step.e2e_bounds) > 1
    step.dlogits.fill_(float("nan"))          # the e2e path must write every row again
    step.e2e_step()
    step.e2e_step()                           # twice: the second step reuses the buffers
    torch.cuda.synchronize()
    for k, v in want.items():
        got = step.h_out[k]
        assert got.shape == v.shape, k
        assert torch.equal(got.view(torch.int16) if got.dtype == torch.bfloat16 else got.view(torch.int32),
                           v.view(torch.int16) if v.dtype == torch.bfloat16 else v.view(torch.int32)), k
    assert step.h2d > 0 and step.d2h >= want["dlogits"].numel() * want["dlogits"].element_size()
