"""Host logic of the vocabulary-parallel form over two gloo ranks on the CPU: the shard
boundaries gathered from the ranks' widths, the all-gather of the shard statistics in
rank order, and which shard offsets reach the kernels.  The kernels themselves are
replaced by recorders (they run on the GPU and are checked by test_vocab_parallel_gpu)."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

WIDTHS = [5, 11]
B, L = 2, 3


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class _Recorder:
    """Stands in for the binding: the shard statistic encodes who made it."""

    @staticmethod
    def grpo_vocab_shard_stats(logits_shard, vocab_start, *, T, idx, mask):
        R = logits_shard.shape[0] * logits_shard.shape[1]
        st = torch.empty(R, 4)
        st[:, 0] = float(vocab_start)
        st[:, 1] = float(logits_shard.shape[-1])
        st[:, 2] = torch.arange(R, dtype=torch.float32)
        st[:, 3] = float(T)
        return st

    @staticmethod
    def grpo_vocab_combine(stats_all, vocab_starts, B_, L_, **kw):
        return {"stats_all": stats_all, "starts": list(vocab_starts), "B": B_, "L": L_, "kw": kw,
                "logp": torch.full((B_ * L_,), -1.0), "lse": torch.full((B_ * L_,), 2.0),
                "p_rest": torch.full((B_ * L_,), 0.25)}

    @staticmethod
    def grpo_loss_bwd_vocab_shard(logits_shard, vocab_start, vocab_total, idx, adv, dloss, logp, lse, p_rest, **kw):
        return {"start": vocab_start, "total": vocab_total, "logp": logp, "lse": lse, "p_rest": p_rest, "kw": kw}


def _worker(rank, world, port, q):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    from rl_fine_tuning_pass_gb300 import vocab_parallel as vp
    vp.kernels = _Recorder
    starts = vp.gather_vocab_starts(WIDTHS[rank])
    shard = torch.zeros(B, L, WIDTHS[rank])
    idx = torch.zeros(B * L, dtype=torch.int64)
    adv = torch.ones(B)
    fwd = vp.grpo_loss_fwd_vocab_parallel(shard, starts, idx, adv, T=0.7, beta=0.0, eps_low=0.2, eps_high=0.28)
    bwd = vp.grpo_loss_bwd_vocab_parallel(shard, starts, idx, adv, torch.ones(B * L), fwd, T=0.7, beta=0.0,
                                          eps_low=0.2, eps_high=0.28)
    try:
        vp.grpo_loss_fwd_vocab_parallel(torch.zeros(B, L, 3), starts, idx, adv, T=0.7, beta=0.0, eps_low=0.2,
                                        eps_high=0.28)
        width_checked = False
    except ValueError:
        width_checked = True
    q.put((rank, starts, fwd["stats_all"].tolist(), fwd["B"], fwd["L"], fwd["kw"]["grpo"],
           bwd["start"], bwd["total"], float(bwd["p_rest"][0]), width_checked))
    dist.barrier()
    dist.destroy_process_group()


def test_vocab_parallel_orchestration_over_two_gloo_ranks():
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
    for rank, starts, stats_all, b, l, grpo, start, total, p_rest, width_checked in res:
        assert starts == [0, 5, 16]
        assert (b, l, grpo) == (B, L, True)
        # the statistics arrive stacked in rank order, each row in place
        for k in range(2):
            for r in range(B * L):
                assert stats_all[k][r][:3] == [float(starts[k]), float(WIDTHS[k]), float(r)]
                assert abs(stats_all[k][r][3] - 0.7) < 1e-6
        assert (start, total) == (starts[rank], 16)
        assert p_rest == 0.25            # the backward gets the merge's p_rest
        assert width_checked             # a shard that does not match vocab_starts is refused
