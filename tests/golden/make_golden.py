"""Writes tests/golden/grpo_small_case.json: a small fixed case with the oracle's outputs.

It calls only the oracle (and numpy for the seeded inputs).  The fixture guards the
oracle against unintended changes; whenever the oracle's arithmetic changes on purpose,
rerun this script and name the passage that justifies the change in the commit.
Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402


def small_case():
    rng = np.random.default_rng(20261202)
    B, L, V = 2, 4, 16
    R = B * L
    x32 = (rng.standard_normal((R, V)) * 2.0).astype(np.float32)
    bits = oracle.round_to_bf16_bits(x32.astype(np.float64))
    x = oracle.bf16_bits_to_fp64(bits)
    idx = rng.integers(0, V, R)
    T, beta, el, eh = 0.9, 0.04, 0.2, 0.28
    logp, _ = oracle.selective_log_softmax(x, idx, T)
    old = (logp + rng.standard_normal(R) * 0.3).astype(np.float32).astype(np.float64)
    ref = (logp + rng.standard_normal(R) * 0.1).astype(np.float32).astype(np.float64)
    A = np.array([0.75, -1.25])
    mask = np.array([1, 1, 1, 0, 1, 1, 0, 0], dtype=np.uint8)
    dloss = mask / np.repeat(mask.reshape(B, L).sum(1) * B, L)
    return dict(B=B, L=L, V=V, T=T, beta=beta, eps_low=el, eps_high=eh, logits_bf16=bits.tolist(),
                idx=idx.tolist(), old_logp=old.tolist(), ref_logp=ref.tolist(), adv=A.tolist(),
                mask=mask.tolist(), dloss=dloss.tolist())


def outputs(case):
    x = oracle.bf16_bits_to_fp64(np.array(case["logits_bf16"], dtype=np.uint16))
    L = case["L"]
    adv = oracle.per_row(case["adv"], L)
    args = (x, np.array(case["idx"]), np.array(case["old_logp"]), np.array(case["ref_logp"]), adv,
            np.array(case["mask"], dtype=np.uint8))
    f = oracle.grpo_loss_fwd(*args, case["T"], case["beta"], case["eps_low"], case["eps_high"])
    dl, g = oracle.grpo_loss_bwd(*args, np.array(case["dloss"]), case["T"], case["beta"],
                                 case["eps_low"], case["eps_high"])
    return dict(loss=f["loss"].tolist(), logp=f["logp"].tolist(), lse=f["lse"].tolist(),
                kl=f["kl"].tolist(), entropy=f["entropy"].tolist(),
                is_clipped=[int(v) for v in f["is_clipped"]], g=g.tolist(),
                dlogits_bf16=oracle.round_to_bf16_bits(dl).tolist())


if __name__ == "__main__":
    case = small_case()
    out = {"_written_by": "tests/golden/make_golden.py (oracle only)", "case": case, "oracle": outputs(case)}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "grpo_small_case.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", path)
