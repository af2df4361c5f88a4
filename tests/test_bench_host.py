"""bench.py host logic on the CPU: byte accounting, whole-job aggregation over ranks
(world size 2 with the gloo backend), and the reference arm's rank handling."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from rl_fine_tuning_pass_gb300 import workloads as W  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    local_ms = [10.0, 25.0][rank]
    total = bench.aggregate_max_ms(local_ms, world, "cpu")
    gbs, rps = bench.whole_job_rates(1_000_000, 64, 10, world, total)
    q.put((rank, total, gbs, rps))
    dist.barrier()
    dist.destroy_process_group()


def test_aggregation_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, total, gbs, rps in res:
        assert total == 25.0                      # max over ranks, on every rank
        assert abs(gbs - 1_000_000 * 10 * 2 / 0.025 / 1e9) < 1e-9
        assert abs(rps - 64 * 10 * 2 / 0.025) < 1e-6


def test_single_rank_aggregation_is_identity():
    assert bench.aggregate_max_ms(7.5, 1, "cpu") == 7.5


def test_grpo_row_bytes_classes():
    spec = W.get("grpo_b4_l512_v32000")
    live = np.array([1, 1, 0, 1], bool)
    zero = np.array([0, 1, 1, 0], bool)
    f, b = bench.grpo_row_bytes(spec, live, zero, has_mask=True, has_old=True, has_ref=False)
    Vs = spec.V * 2
    assert list(f) == [1 + 21 + Vs + 12, 1 + 21 + Vs + 12, 1 + 21, 1 + 21 + Vs + 12]
    # full row: write + read + scalars; zero row: write only (+ its factor inputs); masked: write + mask
    assert list(b) == [1 + Vs + 12 + 12 + Vs, 1 + Vs + 12, 1 + Vs, 1 + Vs + 12 + 12 + Vs]


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_line_shape():
    """Rank 0 of the reference arm: one JSON line with the oracle's throughput (small steps)."""
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "grpo_b4_l512_v32000", "--steps", "2", "--warmup", "0"],
                         capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["config"]["workload"] == "grpo_b4_l512_v32000"
    assert "rows [0, 2048)" in line["cpu_baseline"]["sample"]


def test_default_workload_is_the_largest_single_gpu_config():
    """With no flags the bench times the 20 GB (16, 4096, 151936) GRPO step at beta 0.04 with
    8 of 16 zero-advantage sequences."""
    args = bench.parse_args([])
    spec = bench.make_spec(args)
    assert spec.name == "sweep_b16_l4096_v151936" and (spec.B, spec.L, spec.V) == (16, 4096, 151936)
    assert spec.beta == 0.04 and spec.zero_adv_seqs == 8 and spec.dtype == "bf16"


def test_vocab_shard_starts_cover_the_vocabulary():
    for V, S in [(32000, 4), (151936, 8), (7, 3), (5, 5)]:
        st = bench.vocab_shard_starts(V, S)
        assert st[0] == 0 and st[-1] == V and len(st) == S + 1
        w = np.diff(st)
        assert (w >= 1).all() and w.max() - w.min() <= 1


def test_step_kind_and_sequence_samples():
    """The sequence-level pass is sampled in whole sequences (its ratio sums over one);
    the other passes sample single rows."""
    spec = W.get("grpo_b4_l512_v32000")
    args = bench.parse_args(["--seq-level"])
    assert bench.step_kind(args, spec) == "seq"
    assert bench.step_kind(bench.parse_args([]), spec) == "grpo"
    ent = W.get("entropy_slsm_b16_l4096_v32000")
    assert bench.step_kind(bench.parse_args(["--entropy-bwd"]), ent) == "entropy_bwd"
    assert bench.step_kind(bench.parse_args([]), ent) == "slsm"
    rows = bench.oracle_slice(spec, "seq", 700, 5)
    assert len(rows) == 2 * spec.L and rows[0] % spec.L == 0 and (np.diff(rows) == 1).all()
    big = W.get("sweep_b16_l4096_v151936")
    for kind in ("grpo", "seq"):
        a, b = bench.oracle_slice(big, kind), bench.oracle_slice(big, kind)
        assert np.array_equal(a, b), "the oracle sample is fixed"
        assert (np.diff(a) == 1).all() and 0 <= a[0] and a[-1] < big.rows
    r = bench.oracle_slice(big, "grpo")
    assert len(r) == 2048 and r[0] % 2048 == 0
    assert len(bench.oracle_slice(big, "seq")) == big.L  # one whole sequence


def test_oracle_pool_times_the_same_sample_each_run():
    """Both baseline legs time the oracle through time_oracle: the sample handed over once,
    a warm-up run, then the median of the repeats."""
    spec = W.get("tiny_fp32")
    inp = W.generate(spec, 0)
    import oracle
    rows = np.arange(spec.rows)
    x = inp.logits.reshape(-1, spec.V).double().numpy()
    lp, _ = oracle.selective_log_softmax(x, inp.idx.numpy(), spec.T)
    smp = {"x": x, "idx": inp.idx.numpy(), "adv": oracle.per_row(inp.adv.numpy(), spec.L), "mask": None,
           "old": lp + inp.old_offset.double().numpy(), "ref": lp + inp.ref_offset.double().numpy(),
           "dloss": inp.dloss.double().numpy()}
    med, used, times = bench.time_oracle(spec, "grpo", smp, warmup=1, repeats=3)
    assert len(times) == 3 and med == sorted(times)[1] and used >= 1
    assert bench.sample_bytes(spec, "grpo", smp) > 0
    assert len(rows) == spec.rows


def test_oracle_pool_splits_whole_units_and_runs():
    """The all-cores oracle baseline: parts are disjoint, cover the sample, and keep whole
    sequences for the sequence-level pass; two spawned workers run the oracle on them."""
    import oracle
    spec = W.get("grpo_b4_l512_v32000", B=3, L=8, V=64)
    inp = W.generate(spec, 0, device="cpu")
    x = oracle.bf16_bits_to_fp64(inp.logits.reshape(-1, spec.V).view(torch.int16).numpy().view(np.uint16))
    smp = {"x": x, "idx": inp.idx.numpy(), "adv": oracle.per_row(inp.adv.numpy(), spec.L), "mask": inp.mask.numpy(),
           "old": None, "ref": None, "dloss": inp.dloss.double().numpy(), "adv_seq": inp.adv.double().numpy()}
    for kind, unit in (("grpo", 1), ("seq", spec.L)):
        pool = bench.OraclePool(2, spec, kind)
        try:
            parts = pool.split(smp)
            assert len(parts) == 2
            assert np.array_equal(np.concatenate([p["x"] for p in parts]), x)
            assert all(len(p["idx"]) % unit == 0 for p in parts)
            if kind == "seq":
                assert np.array_equal(np.concatenate([p["adv_seq"] for p in parts]), smp["adv_seq"])
            pool.load(smp)
            assert len(pool.active) == 2
            assert pool.go() > 0 and pool.go() > 0  # the loaded sample runs again
        finally:
            pool.close()


def test_kernel_source_hash_per_entry_point():
    """Each entry point's hash covers its translation units and what they include, and no more."""
    seq = bench._source_closure(bench.KERNEL_UNITS["grpo_seq_terms"])
    assert "rowpass_seq.cu" in seq and "rowpass_common.cuh" in seq and "rowpass_fwd.cuh" not in seq
    fused = bench._source_closure(bench.KERNEL_UNITS["grpo_loss_fused"])
    assert {"rowpass_fused.cuh", "rowpass_fwd.cuh", "rowpass_bwd.cuh", "rowpass_internal.h"} <= set(fused)
    hashes = {k: bench.kernel_source_hash(k) for k in bench.KERNEL_UNITS}
    assert hashes["grpo_loss_fwd"] == hashes["entropy_from_logits"] != hashes["grpo_loss_bwd"]
    assert all(len(h) == 16 for h in hashes.values())
    spec = bench.W.get("grpo_b4_l512_v32000")
    assert bench.measured_traffic("not_an_entry_point", spec) is None
    # a record belongs to its workload's own configuration only
    if bench.measured_traffic("grpo_loss_bwd", spec) is not None:
        assert bench.measured_traffic("grpo_loss_bwd", spec.with_(beta=0.04)) is None
        assert bench.measured_traffic("grpo_loss_bwd", spec.with_(B=2)) is None


def test_e2e_parts_cover_every_row_once():
    """Parts of the end-to-end path: whole sequences where required or when there are
    enough sequences, else token ranges of one sequence; together every row exactly once."""
    for B, L, P, whole in [(4, 512, 16, False), (4, 512, 16, True), (16, 1024, 16, False), (3, 5, 16, False),
                           (1, 7, 4, False), (20, 3, 16, False)]:
        parts = bench.e2e_parts(B, L, P, whole)
        seen = np.zeros(B * L, int)
        for b0, b1, l0, l1 in parts:
            assert 0 <= b0 < b1 <= B and 0 <= l0 < l1 <= L
            assert b1 - b0 == 1 or (l0, l1) == (0, L)      # a token range stays in one sequence
            if whole:
                assert (l0, l1) == (0, L)
            for b in range(b0, b1):
                seen[b * L + l0:b * L + l1] += 1
        assert np.all(seen == 1), (B, L, P, whole)


def test_fused_row_bytes_classes():
    """The fused step reads an unmasked row's logits once and writes every row's dlogits."""
    spec = W.get("grpo_b4_l512_v32000")
    Vs = spec.V * 2
    b = bench.fused_row_bytes(spec, np.array([1, 0], bool), has_mask=True, has_old=True, has_ref=True)
    assert list(b) == [1 + 21 + Vs + Vs + 8 + 4 + 4 + 4, 1 + 21 + Vs]
    b = bench.fused_row_bytes(spec, np.array([1], bool), has_mask=False, has_old=False, has_ref=False)
    assert list(b) == [21 + Vs + Vs + 8 + 4]
