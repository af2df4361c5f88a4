#!/usr/bin/env python3
"""Benchmark of the GRPO row pass on GB300.

One step = one pass of the whole hot path over one batch of synthetic logits:

* GRPO workloads (default ``sweep_b16_l4096_v151936``: B=16, L=4096, V=151936, ~20 GB of
  bf16 logits, T=0.7, beta=0.04, 8 of 16 sequences with advantage 0 -- the largest of the
  Qwen3-vocabulary shapes; ``grpo_b4_l512_v32000`` is the GRPO backward workload of the
  Liger-Kernel GRPO Loss Backward write-up, (B, L, V, zero-grad%) = (4, 512, 32000, 50%)):
  ``grpo_loss_fwd`` (loss, logp, lse, kl, is_clipped, entropy) then ``grpo_loss_bwd``;
  with ``--fused``, the single kernel ``grpo_loss_fused`` (dloss known in advance); with
  ``--seq-level``, the sequence-level form (``selective_log_softmax_fwd``,
  ``grpo_seq_terms``, ``selective_log_softmax_bwd``); with ``--vocab-shards S``, the
  vocabulary-parallel form with its S shards run one after another.  The same line
  carries ``entropy``: ``entropy_from_logits`` timed alone over the same logits, and (for
  the fwd + bwd step) ``fused``: ``grpo_loss_fused`` timed alone over the same batch, with
  its rows/s over the step's.
* ``entropy_slsm_b16_l4096_v32000``: ``entropy_from_logits``, ``selective_log_softmax_fwd``
  and ``selective_log_softmax_bwd``; with ``--entropy-bwd``, ``entropy_from_logits`` (with
  lse) and ``entropy_from_logits_bwd``.
* ``linear_qwen3_b16_l1024_h1024_v151936``: ``grpo_fused_linear`` on hidden states and a
  Qwen3-0.6B-shaped LM head (rows/s and tensor TFLOP/s).

The metric is algorithmic HBM bytes per second (the minimal bytes of the step: each
unmasked row's logits read once by the forward; each backward row with a non-zero
factor read once and written once; each zero row written once; plus the per-row
scalars), and rows per second.  Inputs are resident in HBM when the timed region
starts; L2 is flushed (a 256 MB write, then a 256 MB read so no dirty lines remain)
before every timed step and the flush is not timed.  ``e2e`` repeats the measurement
through the C-ABI entry points with the inputs in pinned host memory and the outputs
copied back, copies inside the timed region.  ``cpu_baseline`` (and ``--impl
reference``) time the fp64 oracle on the host cores over one fixed seeded slice of
2048 rows of the same workload: warm-up runs, then the median of the timed runs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own batch (weak scaling; no collective on the
data path) and rank 0 prints one JSON line with the aggregate over ranks.
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time
import weakref

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from rl_fine_tuning_pass_gb300 import binding as rp  # noqa: E402
from rl_fine_tuning_pass_gb300 import workloads as W  # noqa: E402

METRIC = "GRPO fwd+bwd logits GB/s"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20


class L2Flush:
    """Evicts L2 between timed steps: a 256 MB write (larger than the 129 MB L2), then a
    256 MB read of another buffer so that the written lines are written back during the
    flush and none of the flush's dirty lines are left for the timed kernels to evict."""

    def __init__(self, device):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        # fp32, so that the sum reads the buffer directly (an int32 sum into int64 would
        # first write a 512 MB cast copy)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.sink = torch.empty((), dtype=torch.float32, device=device)

    def __call__(self, i: int = 0):
        self.w.fill_(i & 0x7F)
        torch.sum(self.r, dim=0, out=self.sink)
GRPO_WORKLOADS = ("grpo_b4_l512_v32000", "grpo_qwen3_b16_l1024_v151936", "sweep_b16_l4096_v151936")
LINEAR_WORKLOAD = "linear_qwen3_b16_l1024_h1024_v151936"
LINEAR_METRIC = "GRPO loss on the LM head (fused linear) rows/s"


# ---------------------------------------------------------------------------
# environment
# ---------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_bf16_peak(sustained=True):
    """The measured dense bf16 tensor peak (TFLOP/s): the sustained figure for work timed
    inside a long loop, else the burst figure."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        k = "bf16_tflops_sustained" if sustained else "bf16_tflops"
        return float(p[k]), f"measured (MEASURED_PEAKS.json {k}, cuBLAS bf16 GEMM)"
    except Exception:
        return (1700.0 if sustained else 1900.0), "fallback (no MEASURED_PEAKS.json)"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


# Translation units behind each entry point; with the files they include (closure of the
# quoted #include lines) they fix that entry point's kernels and launch shapes.
_FWD = ("rowpass_fwd_bf16.cu", "rowpass_fwd_f32.cu")
_BWD = ("rowpass_bwd_bf16.cu", "rowpass_bwd_f32.cu")
KERNEL_UNITS = {
    "grpo_loss_fwd": _FWD, "entropy_from_logits": _FWD, "selective_log_softmax_fwd": _FWD,
    "grpo_vocab_shard_stats": _FWD,
    "grpo_loss_bwd": _BWD, "selective_log_softmax_bwd": _BWD, "entropy_from_logits_bwd": _BWD,
    "grpo_loss_bwd_vocab_shard": _BWD,
    "grpo_loss_fused": ("rowpass_fused_bf16.cu", "rowpass_fused_f32.cu"),
    "grpo_seq_terms": ("rowpass_seq.cu",),
    "grpo_vocab_combine": ("rowpass_vocab.cu",),
    "grpo_fused_linear": ("rowpass_linear.cu",),
}


def _source_closure(units):
    csrc = os.path.join(ROOT, "rl_fine_tuning_pass_gb300", "csrc")
    search = (csrc, os.path.join(ROOT, "include"))
    seen, todo = {}, list(units)
    while todo:
        name = todo.pop()
        if name in seen:
            continue
        path = next((os.path.join(d, name) for d in search if os.path.isfile(os.path.join(d, name))), None)
        if path is None:
            continue
        with open(path, "rb") as f:
            seen[name] = f.read()
        for line in seen[name].decode(errors="replace").splitlines():
            line = line.strip()
            if line.startswith("#include \""):
                todo.append(line.split('"')[1])
    return seen


def kernel_source_hash(kernel: str = None) -> str:
    """Hash of the kernel sources: all of them, or those behind one entry point."""
    if kernel is None:
        csrc = os.path.join(ROOT, "rl_fine_tuning_pass_gb300", "csrc")
        files = {n: open(os.path.join(csrc, n), "rb").read() for n in os.listdir(csrc)}
    else:
        files = _source_closure(KERNEL_UNITS[kernel])
    h = hashlib.sha256()
    for name in sorted(files):
        h.update(name.encode() + b"\0" + files[name])
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, spec):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current sources of that kernel (kernel_source_hash(kernel)) and the workload runs
    with its own configuration (the records are for that one: another beta, batch or
    layout moves other bytes); else None."""
    if spec != W.get(spec.name):
        return None
    workload = spec.name
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    ent = rec.get(workload, {}).get(kernel)
    if not ent or kernel not in KERNEL_UNITS or ent.get("source_hash") != kernel_source_hash(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.sel = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            parts = [p for p in vis.split(",") if p.strip()]
            self.sel = parts[device_index] if device_index < len(parts) else str(device_index)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", self.sel], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            n += 1
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": n}


# ---------------------------------------------------------------------------
# workloads: prebuilt C-ABI calls with preallocated outputs
# ---------------------------------------------------------------------------

def _p(t):
    return None if t is None else t.data_ptr()


def grpo_row_bytes(spec, live, zero_g, has_mask, has_old, has_ref):
    """Minimal bytes per row of the GRPO forward and backward (numpy bool arrays in,
    int arrays out).  Forward: an unmasked row reads its V logits, idx, old/ref; every
    row reads its mask byte and writes loss, logp, lse, kl, entropy (4 B each) and
    is_clipped (1 B).  Backward: every row reads its mask byte and writes V dlogits; an
    unmasked row reads logp, old, ref, dloss; a row with a non-zero factor also reads
    idx, lse and its V logits.  The per-sequence advantages (4 B each) are left out."""
    V, s = spec.V, spec.elem_size
    live = np.asarray(live, bool)
    zero_g = np.asarray(zero_g, bool)
    m = 1 if has_mask else 0
    o = 4 if has_old else 0
    r = 4 if has_ref else 0
    fwd = m + 21 + live * (V * s + 8 + o + r)
    bwd = m + V * s + live * (4 + o + r + 4) + (~zero_g) * (8 + 4 + V * s)
    return fwd.astype(np.int64), bwd.astype(np.int64)


def fused_row_bytes(spec, live, has_mask, has_old, has_ref):
    """Minimal bytes per row of the fused forward + backward: an unmasked row reads its V
    logits once (and idx, old, ref, dloss), every row reads its mask byte, writes the
    forward outputs (21 B) and its V dlogits."""
    V, s = spec.V, spec.elem_size
    live = np.asarray(live, bool)
    m = 1 if has_mask else 0
    o = 4 if has_old else 0
    r = 4 if has_ref else 0
    return (m + 21 + V * s + live * (V * s + 8 + o + r + 4)).astype(np.int64)


SLSM_ROW_BYTES = {"entropy_from_logits": lambda V, s: V * s + 4,
                  "selective_log_softmax_fwd": lambda V, s: V * s + 8 + 8,
                  "selective_log_softmax_bwd": lambda V, s: 2 * V * s + 8 + 4 + 4}


def _unregister_host(ptr):
    torch.cuda.cudart().cudaHostUnregister(ptr)


def pinned_host(shape, dtype, src=None):
    """A page-locked host tensor, filled from ``src`` if given.

    Inputs (src given) come from the CUDA host allocator (cudaHostAlloc; torch rounds the
    block up to a power of two), outputs are malloc'd pages registered with cudaHostRegister
    at exactly their size.  On GB300 machines each kind kept its full copy rate in its own
    direction after a long-running process had churned the host memory (20 GB host->device
    from registered pages dropped to ~12 GB/s there, from cudaHostAlloc's it did not; the
    reverse held for device->host), while on a fresh box both are at ~190-210 GB/s."""
    if src is not None:
        t = torch.empty(shape, dtype=dtype, pin_memory=True)
        t.copy_(src)
        return t
    t = torch.empty(shape, dtype=dtype)
    nbytes = t.numel() * t.element_size()
    if nbytes and int(torch.cuda.cudart().cudaHostRegister(t.data_ptr(), nbytes, 0)) == 0:
        weakref.finalize(t, _unregister_host, t.data_ptr())
    elif nbytes:
        t = t.pin_memory()
    return t


def host_memory_available() -> int:
    """Bytes this process may still take: MemAvailable, capped by the cgroup's limit."""
    avail = None
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    avail = int(line.split()[1]) * 1024
    except OSError:
        pass
    for lim_p, use_p in (("/sys/fs/cgroup/memory.max", "/sys/fs/cgroup/memory.current"),
                         ("/sys/fs/cgroup/memory/memory.limit_in_bytes", "/sys/fs/cgroup/memory/memory.usage_in_bytes")):
        try:
            with open(lim_p) as f:
                lim = f.read().strip()
            with open(use_p) as f:
                use = int(f.read().strip())
            if lim != "max" and int(lim) < (1 << 60):
                left = int(lim) - use
                avail = left if avail is None else min(avail, left)
            break
        except (OSError, ValueError):
            continue
    return avail if avail is not None else 1 << 62


class PipelinedE2E:
    """End-to-end through the public API with host buffers.  The batch is cut into parts: a
    part is a group of whole sequences, or, for the token-level passes when there are
    fewer sequences than parts, a range of one sequence's tokens (the public calls take it
    as a batch of one sequence of that many tokens).  The per-row and per-sequence inputs
    go host -> device once at the start of the step; then each part's logits go host ->
    device on one stream, its calls run on a second once they have landed, and its outputs
    go device -> host on a third, so the two copy directions and the kernels of
    neighbouring parts overlap.  A subclass names its inputs (e2e_inputs: tensor and
    layout: "bl" = [B, L, ...], "s" = one value per sequence, "r" = one value per row), its
    outputs (e2e_outputs: shape, dtype, layout) and makes the public calls of one part
    (e2e_part)."""

    E2E_PARTS = 16               # at most; parts of at least E2E_PART_BYTES of logits
    E2E_PART_BYTES = 32 << 20    # below this the calls' host-side cost outweighs a part's copy time
    E2E_WHOLE_SEQUENCES = False  # True where a part must hold whole sequences
    E2E_VIEWS = True             # e2e_part takes the part's input views (False: it has its own)

    def e2e_setup(self):
        dev = self.inp.logits.device
        ins = {k: v for k, v in self.e2e_inputs().items() if v[0] is not None}
        outs = self.e2e_outputs()
        # the step's per-element outputs (dlogits) come back too when the host has room for
        # them beside the inputs; else only the per-row results (loss ...) do
        nb = lambda shape, dt: math.prod(shape) * torch.empty((), dtype=dt).element_size()
        in_bytes = sum(t.numel() * t.element_size() for t, _ in ins.values())
        out_bytes = sum(nb(shape, dt) for shape, dt, _ in outs.values())
        self.e2e_outputs_kept = "all"
        if in_bytes + out_bytes > 0.5 * host_memory_available():
            outs = {k: v for k, v in outs.items() if v[2] != "bl"}
            self.e2e_outputs_kept = "per-row results only (the host has no room for the per-element outputs)"
        self.h_in = {k: pinned_host(t.shape, t.dtype, src=t) for k, (t, _) in ins.items()}
        self.d_in = {k: torch.empty(t.shape, dtype=t.dtype, device=dev) for k, (t, _) in ins.items()}
        self.lay_in = {k: lay for k, (_, lay) in ins.items()}
        self.h_out = {k: pinned_host(shape, dt) for k, (shape, dt, _) in outs.items()}
        self.lay_out = {k: lay for k, (_, _, lay) in outs.items()}
        self.h2d = sum(t.numel() * t.element_size() for t in self.h_in.values())
        self.d2h = sum(t.numel() * t.element_size() for t in self.h_out.values())
        logit_bytes = self.h_in["logits"].numel() * self.h_in["logits"].element_size()
        n = int(max(1, min(self.E2E_PARTS, (logit_bytes + self.E2E_PART_BYTES // 2) // self.E2E_PART_BYTES)))
        self.e2e_bounds = e2e_parts(self.spec.B, self.spec.L, n, self.E2E_WHOLE_SEQUENCES)
        self.e2e_streams = [torch.cuda.Stream(device=dev) for _ in range(3)]
        # the per-part copy-in views, made once
        self.e2e_in_views = [[(self._cut(self.d_in[k], "bl", part), self._cut(h, "bl", part))
                              for k, h in self.h_in.items() if self.lay_in[k] == "bl"] for part in self.e2e_bounds]

    def _cut(self, t, lay, part):
        b0, b1, l0, l1 = part
        if lay == "bl":
            return t[b0:b1, l0:l1]
        if lay == "s":
            return t[b0:b1]
        L = self.spec.L
        return t[b0 * L + l0:(b1 - 1) * L + l1]

    def e2e_step(self):
        s_in, s_run, s_out = self.e2e_streams
        main = torch.cuda.current_stream()
        s_in.wait_stream(main)  # the previous step is over (main waited for its last copy out)
        landed = []
        with torch.cuda.stream(s_in):
            for k, h in self.h_in.items():  # per-row and per-sequence inputs: once per step
                if self.lay_in[k] != "bl":
                    self.d_in[k].copy_(h, non_blocking=True)
            for views in self.e2e_in_views:
                for dst, src in views:
                    dst.copy_(src, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(s_in)
                landed.append(ev)
        done = []
        with torch.cuda.stream(s_run):
            for part, ev in zip(self.e2e_bounds, landed):
                s_run.wait_event(ev)
                d = {k: self._cut(t, self.lay_in[k], part) for k, t in self.d_in.items()} if self.E2E_VIEWS else None
                out = self.e2e_part(d, part)
                ev2 = torch.cuda.Event()
                ev2.record(s_run)
                done.append((ev2, out))
        with torch.cuda.stream(s_out):
            for part, (ev, out) in zip(self.e2e_bounds, done):
                s_out.wait_event(ev)
                for k, t in out.items():
                    if k not in self.h_out:
                        continue
                    t.record_stream(s_out)  # allocated on s_run, read here
                    self._cut(self.h_out[k], self.lay_out[k], part).copy_(t, non_blocking=True)
        main.wait_stream(s_out)

    def e2e_part(self, d, part):
        raise NotImplementedError


def e2e_parts(B, L, P, whole_sequences):
    """Parts (b0, b1, l0, l1) of a batch of B sequences of L tokens: P groups of whole
    sequences when B >= P (or when whole sequences are required), else every sequence cut
    into ceil(P / B) token ranges."""
    if whole_sequences or B >= P:
        n = max(1, min(B, P))
        return [(B * k // n, B * (k + 1) // n, 0, L) for k in range(n)]
    per = min(L, -(-P // B))
    return [(b, b + 1, L * k // per, L * (k + 1) // per) for b in range(B) for k in range(per)]


class GrpoStep(PipelinedE2E):
    """grpo_loss_fwd (+entropy, kl, is_clipped) then grpo_loss_bwd over one batch."""

    oracle_kind = "grpo"
    E2E_PART_BYTES = 16 << 20  # its e2e calls go through the C ABI (e2e_setup)

    def __init__(self, spec, seed, device, inputs=None):
        self.spec = spec
        lib = rp.load_library()
        inp = inputs if inputs is not None else W.generate(spec, seed, device=device)
        self.inp = inp
        T, beta = spec.T, spec.beta
        R = spec.rows
        # old/ref placed near the current logp with our own forward (setup, not timed)
        logp0, _ = rp.selective_log_softmax_fwd(inp.logits, inp.idx, T=T)
        self.old = (logp0 + inp.old_offset).contiguous() if inp.old_offset is not None else None
        self.ref = (logp0 + inp.ref_offset).contiguous() if (inp.ref_offset is not None and beta != 0) else None
        f32 = dict(dtype=torch.float32, device=device)
        self.out = {k: torch.empty(R, **f32) for k in ("loss", "logp", "lse", "kl", "entropy")}
        self.out["is_clipped"] = torch.empty(R, dtype=torch.uint8, device=device)
        self.dlogits = torch.empty(inp.logits.shape, dtype=inp.logits.dtype, device=device)
        self.x_desc = rp.rows_of(inp.logits)
        self.dx_desc = rp.rows_of(self.dlogits)
        self.stream = torch.cuda.current_stream(device).cuda_stream
        o = self.out
        self._fwd = lib.grpo_loss_fwd
        self._bwd = lib.grpo_loss_bwd
        self.fwd_args = (ctypes.byref(self.x_desc), _p(inp.idx), _p(self.old), _p(self.ref), _p(inp.adv),
                         _p(inp.mask), T, beta, spec.eps_low, spec.eps_high, _p(o["loss"]), _p(o["logp"]),
                         _p(o["lse"]), _p(o["kl"]), _p(o["is_clipped"]), _p(o["entropy"]), None, self.stream)
        self.bwd_args = (ctypes.byref(self.x_desc), _p(inp.idx), _p(self.old), _p(self.ref), _p(inp.adv),
                         _p(inp.mask), _p(inp.dloss), _p(o["logp"]), _p(o["lse"]), T, beta, spec.eps_low,
                         spec.eps_high, ctypes.byref(self.dx_desc), None, self.stream)
        self.kernels = [("grpo_loss_fwd", self.fwd), ("grpo_loss_bwd", self.bwd)]

    def fwd(self):
        st = self._fwd(*self.fwd_args)
        if st:
            raise rp.GrpoError("grpo_loss_fwd", st)

    def bwd(self):
        st = self._bwd(*self.bwd_args)
        if st:
            raise rp.GrpoError("grpo_loss_bwd", st)

    def account(self):
        """Minimal bytes per launch from the row classes of this batch (after one step):
        masked rows, rows whose backward factor is exactly zero, and the rest.  The zero
        factor is read off the inputs and the forward's is_clipped output: with beta == 0
        a row's factor is zero iff it is masked, its dloss is 0, A == 0, or clipping binds."""
        spec, inp = self.spec, self.inp
        R = spec.rows
        mask = torch.ones(R, dtype=torch.bool, device=inp.idx.device) if inp.mask is None else inp.mask.bool()
        adv_row = inp.adv.repeat_interleave(spec.L)
        zero = ~mask | (inp.dloss == 0)
        if spec.beta == 0:
            zero = zero | (adv_row == 0) | self.out["is_clipped"].bool()
        live, zero = mask.cpu().numpy(), zero.cpu().numpy()
        fwd, bwd = grpo_row_bytes(spec, live, zero, inp.mask is not None, self.old is not None, self.ref is not None)
        n_zero = int(zero.sum())
        self.classes = {"rows": R, "masked": int(R - live.sum()), "zero_grad_rows": n_zero,
                        "zero_grad_frac": round(n_zero / R, 4)}
        return {"grpo_loss_fwd": int(fwd.sum()), "grpo_loss_bwd": int(bwd.sum())}

    # -- end-to-end through the public API with host buffers (PipelinedE2E) ------
    def e2e_inputs(self):
        inp = self.inp
        return {"logits": (inp.logits, "bl"), "idx": (inp.idx, "r"), "adv": (inp.adv, "s"), "mask": (inp.mask, "r"),
                "dloss": (inp.dloss, "r"), "old": (self.old, "r"), "ref": (self.ref, "r")}

    def e2e_outputs(self):
        return {"dlogits": (tuple(self.dlogits.shape), self.dlogits.dtype, "bl"),
                "loss": ((self.spec.rows,), torch.float32, "r")}

    def e2e_setup(self):
        """The Python-API calls cost ~0.1 ms of host time a part; through the C ABI with the
        outputs allocated once and each part's arguments made here, a part costs a few
        microseconds, so the batch can be cut into parts of 16 MB."""
        super().e2e_setup()
        if type(self).e2e_part is not GrpoStep.e2e_part:
            return  # a subclass with its own calls
        spec, R = self.spec, self.spec.rows
        dev = self.d_in["logits"].device
        f32 = dict(dtype=torch.float32, device=dev)
        self.e2e_dev_out = {k: torch.empty(R, **f32) for k in ("loss", "logp", "lse", "kl", "entropy")}
        self.e2e_dev_out["is_clipped"] = torch.empty(R, dtype=torch.uint8, device=dev)
        s_run = self.e2e_streams[1].cuda_stream
        T, beta, el, eh = spec.T, spec.beta, spec.eps_low, spec.eps_high
        self.e2e_calls = {}
        for part in self.e2e_bounds:
            x, dx = self._cut(self.d_in["logits"], "bl", part), self._cut(self.dlogits, "bl", part)
            xd, dxd = rp.rows_of(x), rp.rows_of(dx)
            g = lambda k: _p(self._cut(self.d_in[k], self.lay_in[k], part)) if k in self.d_in else None
            o = {k: self._cut(v, "r", part) for k, v in self.e2e_dev_out.items()}
            fa = (ctypes.byref(xd), g("idx"), g("old"), g("ref"), g("adv"), g("mask"), T, beta, el, eh, _p(o["loss"]),
                  _p(o["logp"]), _p(o["lse"]), _p(o["kl"]), _p(o["is_clipped"]), _p(o["entropy"]), None, s_run)
            ba = (ctypes.byref(xd), g("idx"), g("old"), g("ref"), g("adv"), g("mask"), g("dloss"), _p(o["logp"]),
                  _p(o["lse"]), T, beta, el, eh, ctypes.byref(dxd), None, s_run)
            self.e2e_calls[part] = (xd, dxd, fa, ba, {"dlogits": dx, "loss": o["loss"]})
        self.E2E_VIEWS = False

    def e2e_part(self, d, part):
        if d is None:  # the C-ABI path set up in e2e_setup
            _, _, fa, ba, out = self.e2e_calls[part]
            st = self._fwd(*fa)
            if st:
                raise rp.GrpoError("grpo_loss_fwd", st)
            st = self._bwd(*ba)
            if st:
                raise rp.GrpoError("grpo_loss_bwd", st)
            return out
        spec = self.spec
        f = rp.grpo_loss_fwd(d["logits"], d["idx"], d["adv"], T=spec.T, beta=spec.beta, eps_low=spec.eps_low,
                             eps_high=spec.eps_high, old_logp=d.get("old"), ref_logp=d.get("ref"), mask=d.get("mask"),
                             with_entropy=True)
        dl = rp.grpo_loss_bwd(d["logits"], d["idx"], d["adv"], d["dloss"], f["logp"], f["lse"], T=spec.T,
                              beta=spec.beta, eps_low=spec.eps_low, eps_high=spec.eps_high, old_logp=d.get("old"),
                              ref_logp=d.get("ref"), mask=d.get("mask"),
                              dlogits=self._cut(self.dlogits, "bl", part))
        return {"dlogits": dl, "loss": f["loss"]}


class FusedStep(GrpoStep):
    """grpo_loss_fused: forward outputs and dlogits in one kernel (dloss known in advance)."""

    E2E_PART_BYTES = 32 << 20  # public Python API calls per part

    def __init__(self, spec, seed, device, inputs=None):
        super().__init__(spec, seed, device, inputs)
        lib = rp.load_library()
        inp, o = self.inp, self.out
        self._fused = lib.grpo_loss_fused
        self.fused_args = (ctypes.byref(self.x_desc), _p(inp.idx), _p(self.old), _p(self.ref), _p(inp.adv),
                           _p(inp.mask), _p(inp.dloss), spec.T, spec.beta, spec.eps_low, spec.eps_high,
                           _p(o["loss"]), _p(o["logp"]), _p(o["lse"]), _p(o["kl"]), _p(o["is_clipped"]),
                           _p(o["entropy"]), ctypes.byref(self.dx_desc), None, self.stream)
        self.kernels = [("grpo_loss_fused", self.fused)]

    def fused(self):
        st = self._fused(*self.fused_args)
        if st:
            raise rp.GrpoError("grpo_loss_fused", st)

    def account(self):
        spec, inp = self.spec, self.inp
        R = spec.rows
        live = np.ones(R, bool) if inp.mask is None else inp.mask.bool().cpu().numpy()
        b = fused_row_bytes(spec, live, inp.mask is not None, self.old is not None, self.ref is not None)
        zero = (~torch.from_numpy(live).to(inp.idx.device)) | (inp.dloss == 0)
        if spec.beta == 0:
            zero = zero | (inp.adv.repeat_interleave(spec.L) == 0) | self.out["is_clipped"].bool()
        n_zero = int(zero.sum())
        self.classes = {"rows": R, "masked": int(R - live.sum()), "zero_grad_rows": n_zero,
                        "zero_grad_frac": round(n_zero / R, 4), "fused": True}
        return {"grpo_loss_fused": int(b.sum())}

    def e2e_part(self, d, part):
        spec = self.spec
        f = rp.grpo_loss_fused(d["logits"], d["idx"], d["adv"], d["dloss"], T=spec.T, beta=spec.beta,
                               eps_low=spec.eps_low, eps_high=spec.eps_high, old_logp=d.get("old"),
                               ref_logp=d.get("ref"), mask=d.get("mask"), with_entropy=True,
                               dlogits=self._cut(self.dlogits, "bl", part))
        return {"dlogits": f["dlogits"], "loss": f["loss"]}


class LinearStep:
    """grpo_fused_linear over the LM-head workload: per chunk of rows, the logits GEMM,
    the row pass, the hidden-state gradient GEMM and the head-weight gradient GEMM."""

    def __init__(self, spec, seed, device, chunk_rows):
        self.spec = spec
        li = W.generate_linear(spec, seed, device=device)
        self.li = li
        self.chunk = min(chunk_rows, spec.rows)
        R, V, H = spec.rows, spec.V, spec.H
        f32 = dict(dtype=torch.float32, device=device)
        self.grad_w = torch.zeros(V, H, **f32)
        self.ws = torch.empty(rp.grpo_fused_linear_workspace_size(H, V, self.chunk), dtype=torch.uint8, device=device)
        # old / ref placed near the current logp with a first pass of the same call (setup)
        f0 = rp.grpo_fused_linear(li.hidden, li.weight, li.idx, li.adv, li.dloss, B=spec.B, L=spec.L, T=spec.T,
                                  beta=0.0, eps_low=spec.eps_low, eps_high=spec.eps_high, mask=li.mask,
                                  chunk_rows=self.chunk, with_grad_hidden=False, with_grad_weight=False,
                                  workspace=self.ws)
        self.old = (f0["logp"] + li.old_offset).contiguous()
        self.ref = (f0["logp"] + li.ref_offset).contiguous()
        del f0
        self.kernels = [("grpo_fused_linear", self.call)]
        self.launches_per_step = 7 * ((R + self.chunk - 1) // self.chunk) + (li.mask is not None)
        # the GEMMs run on the unmasked rows only (masked rows are left out of the chunks)
        self.rows_computed = R if li.mask is None else int(li.mask.sum().item())
        self.flops_per_step = 6 * self.rows_computed * V * H

    def call(self, hidden=None, idx=None, adv=None, dloss=None, mask=None, old=None, ref=None):
        spec, li = self.spec, self.li
        pick = lambda a, b: b if a is None else a
        return rp.grpo_fused_linear(pick(hidden, li.hidden), li.weight, pick(idx, li.idx), pick(adv, li.adv),
                                    pick(dloss, li.dloss), B=spec.B, L=spec.L, T=spec.T, beta=spec.beta,
                                    eps_low=spec.eps_low, eps_high=spec.eps_high, old_logp=pick(old, self.old),
                                    ref_logp=pick(ref, self.ref), mask=pick(mask, li.mask), chunk_rows=self.chunk,
                                    grad_weight=self.grad_w, workspace=self.ws)

    def e2e_setup(self):
        li = self.li
        pin = lambda t: None if t is None else t.detach().cpu().pin_memory()
        self.h = {"hidden": pin(li.hidden), "idx": pin(li.idx), "adv": pin(li.adv), "mask": pin(li.mask),
                  "dloss": pin(li.dloss), "old": pin(self.old), "ref": pin(self.ref)}
        R, H = self.spec.rows, self.spec.H
        self.h_gh = torch.empty(R, H, dtype=torch.float32).pin_memory()
        self.h_loss = torch.empty(R, dtype=torch.float32).pin_memory()
        self.h2d = sum(t.numel() * t.element_size() for t in self.h.values() if t is not None)
        self.d2h = self.h_gh.numel() * 4 + self.h_loss.numel() * 4

    def e2e_step(self):
        dev = self.li.hidden.device
        up = {k: None if t is None else t.to(dev, non_blocking=True) for k, t in self.h.items()}
        out = self.call(**up)
        self.h_gh.copy_(out["grad_hidden"], non_blocking=True)
        self.h_loss.copy_(out["loss"], non_blocking=True)


def run_linear(args):
    """Bench line of the LM-head workload: rows/s of the batch and the tensor-core roofline
    of the step (6 R V H flops over its R unmasked rows: the logits GEMM and the two gradient
    GEMMs; masked rows are left out of the chunks)."""
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
    spec = W.get(LINEAR_WORKLOAD, **({"B": args.batch} if args.batch is not None else {}))
    step = LinearStep(spec, args.seed + rank, device, args.chunk_rows)
    flush_buf = L2Flush(device)
    step.call()
    torch.cuda.synchronize()
    K = args.steps if args.steps is not None else 20
    Wm = max(3, args.warmup)
    clocks = ClockSampler(local)
    clocks.start()
    steps, wall = timed_run(step, K, Wm, flush_buf, world, per_kernel=False)
    clk = clocks.stop()
    step_ms = statistics.mean(steps["step"])
    total_ms = aggregate_max_ms(sum(steps["step"]), world, device)
    rows_per_s = spec.rows * K * world / (total_ms * 1e-3)
    peak, peak_src = load_bf16_peak(sustained=True)
    tflops = step.flops_per_step / (step_ms * 1e-3) / 1e12
    e2e = None
    if not args.no_e2e:
        ms = aggregate_max_ms(e2e_run(step, min(K, 10), 2), world, device)  # the slowest rank
        e2e = {"value": round(spec.rows * world / (ms * 1e-3), 1), "unit": "rows/s", "h2d_bytes_per_step": int(step.h2d),
               "d2h_bytes_per_step": int(step.d2h), "ms_per_step": round(ms, 4),
               "path": "public Python API, pinned host hidden states and per-row inputs, loss and grad_hidden "
                       "copied back; the head weight and its gradient stay on the device"}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = linear_cpu_baseline(step)
    if rank == 0:
        full_logits = spec.rows * spec.V * 2
        line = {"metric": LINEAR_METRIC, "unit": "rows/s", "n_gpus": world, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "data": "synthetic",
                "config": {"workload": spec.name, "B": spec.B, "L": spec.L, "H": spec.H, "V": spec.V, "T": spec.T,
                           "beta": spec.beta, "eps_low": spec.eps_low, "eps_high": spec.eps_high,
                           "chunk_rows": step.chunk, "operands": "bf16 hidden and head weight; fp32 accumulation; per chunk, fp16 exponentials of the logits relative to each 128-column maximum, turned into bf16 dlogits in place",
                           "l2": "flushed before every timed step (256 MB write + 256 MB read, not timed)",
                           "parallelism": f"{world} independent batch(es), one per GPU"},
                "value": round(rows_per_s, 1), "steps": K, "warmup": Wm, "ms_per_step": round(step_ms, 4),
                "dtype": "bf16", "rows_per_s": round(rows_per_s, 1),
                "rows_unmasked": step.rows_computed,
                "roofline": {"bound": "tensor", "kernel": "grpo_fused_linear (3 GEMMs + row pass per chunk)",
                             "achieved": round(tflops, 1), "peak": peak, "unit": "TFLOP/s",
                             "frac": round(tflops / peak, 4), "traffic": None, "peak_source": peak_src,
                             "flops_per_step": int(step.flops_per_step)},
                "memory": {"workspace_bytes": int(step.ws.numel()), "full_batch_logits_bytes_bf16": int(full_logits),
                           "full_batch_logits_and_dlogits_bytes_bf16": int(2 * full_logits)},
                "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": step.launches_per_step * K,
                "gpu_launches_note": "once: the masked rows' zero outputs; per chunk (sized for an unmasked "
                                     "batch; chunks past the last unmasked row return at once): the row "
                                     "selection, the gather of the chunk's hidden rows, the logits GEMM, the row "
                                     "pass, grad_hidden's split GEMM and the sum of its splits, the grad_weight "
                                     "GEMM (all this library's kernels)",
                "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"],
                           "samples": clk["samples"]},
                "timed_wall_s": round(wall, 3), "kernel_source": kernel_source_hash()}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def linear_cpu_baseline(step, budget_s=12.0):
    """The oracle's fused_linear_grpo on a bounded sample of rows (the whole head weight)."""
    import oracle
    spec, li = step.spec, step.li
    Wf = oracle.bf16_bits_to_fp64(li.weight.cpu().view(torch.int16).numpy().view(np.uint16))
    def run(n):
        rows = W.sample_rows(spec.rows, n, 13)
        r = torch.as_tensor(rows, device=li.hidden.device)
        hf = oracle.bf16_bits_to_fp64(li.hidden[r].cpu().view(torch.int16).numpy().view(np.uint16))
        g = lambda t: None if t is None else t[r].double().cpu().numpy()
        adv = oracle.per_row(li.adv.cpu().numpy(), spec.L)[rows]
        t0 = time.perf_counter()
        oracle.fused_linear_grpo(hf, Wf, li.idx[r].cpu().numpy(), g(step.old), g(step.ref), adv, g(li.mask),
                                 g(li.dloss), spec.T, spec.beta, spec.eps_low, spec.eps_high)
        return len(rows), time.perf_counter() - t0
    run(4)                      # warm: the first fp64 GEMM call pays the BLAS start-up
    n, dt = run(4)
    n = int(max(4, min(512, budget_s / max(dt / n, 1e-9))))
    n, dt = run(n)
    return {"value": round(n / dt, 3), "unit": "rows/s", "cores": torch.get_num_threads(), "kind": "oracle",
            "sample": f"{n} of {spec.rows} rows of {spec.name} (fp64 numpy, the full head weight), {dt:.1f} s"}


def vocab_shard_starts(V, shards):
    """Boundaries of `shards` near-equal column shards of a V-column vocabulary."""
    return [V * k // shards for k in range(shards + 1)]


class VocabShardStep(GrpoStep):
    """The vocabulary-parallel GRPO step of `shards` ranks, run on one GPU shard after
    shard: grpo_vocab_shard_stats on every shard (each writes its slot of the gathered
    [shards, B*L, 4] buffer, where an all-gather would put it), grpo_vocab_combine, then
    grpo_loss_bwd_vocab_shard on every shard into its columns of dlogits."""

    E2E_PART_BYTES = 32 << 20  # public Python API calls per part

    def __init__(self, spec, seed, device, shards, inputs=None):
        super().__init__(spec, seed, device, inputs)
        lib = rp.load_library()
        inp, o, R, V = self.inp, self.out, spec.rows, spec.V
        self.shards = shards
        self.starts = vocab_shard_starts(V, shards)
        self.c_starts = (ctypes.c_int64 * (shards + 1))(*self.starts)
        self.stats = torch.empty(shards, R, 4, dtype=torch.float32, device=device)
        self.p_rest = torch.empty(R, dtype=torch.float32, device=device)
        sl = lambda t, k: t[..., self.starts[k]:self.starts[k + 1]]
        self.x_sh = [rp.rows_of(sl(inp.logits, k)) for k in range(shards)]
        self.dx_sh = [rp.rows_of(sl(self.dlogits, k)) for k in range(shards)]
        T, beta, el, eh = spec.T, spec.beta, spec.eps_low, spec.eps_high
        self._st, self._cb, self._bw = lib.grpo_vocab_shard_stats, lib.grpo_vocab_combine, lib.grpo_loss_bwd_vocab_shard
        self.st_args = [(ctypes.byref(self.x_sh[k]), self.starts[k], _p(inp.idx), _p(inp.mask), T,
                         self.stats[k].data_ptr(), self.stream) for k in range(shards)]
        self.cb_args = (shards, _p(self.stats), self.c_starts, spec.B, spec.L, _p(inp.idx), _p(self.old), _p(self.ref),
                        _p(inp.adv), _p(inp.mask), T, beta, el, eh, _p(o["loss"]), _p(o["logp"]), _p(o["lse"]),
                        _p(o["kl"]), _p(o["is_clipped"]), _p(o["entropy"]), _p(self.p_rest), None, self.stream)
        self.bw_args = [(ctypes.byref(self.x_sh[k]), self.starts[k], V, _p(inp.idx), _p(self.old), _p(self.ref),
                         _p(inp.adv), _p(inp.mask), _p(inp.dloss), _p(o["logp"]), _p(o["lse"]), _p(self.p_rest), T,
                         beta, el, eh, ctypes.byref(self.dx_sh[k]), None, self.stream) for k in range(shards)]
        self.kernels = [("grpo_vocab_shard_stats", self.stats_all_shards), ("grpo_vocab_combine", self.combine),
                        ("grpo_loss_bwd_vocab_shard", self.bwd_all_shards)]
        self.launches_per_step = 2 * shards + 1

    @staticmethod
    def _call(fn, args):
        st = fn(*args)
        if st:
            raise rp.GrpoError(fn.__name__, st)

    def stats_all_shards(self):
        for a in self.st_args:
            self._call(self._st, a)

    def combine(self):
        self._call(self._cb, self.cb_args)

    def bwd_all_shards(self):
        for a in self.bw_args:
            self._call(self._bw, a)

    def account(self):
        """Minimal bytes.  Shard statistics: the logits of every unmasked row once over all
        shards; every shard reads each row's mask byte and writes its 16-byte statistic,
        and reads idx on unmasked rows.  Merge: every row's mask and outputs (21 B) and
        p_rest; an unmasked row's S statistics, idx, old, ref.  Shard backward: the unsplit
        backward's bytes (grpo_row_bytes), its per-row scalars read by every shard, and
        p_rest read by every shard on rows with a non-zero factor."""
        per = super().account()
        spec, inp, S, R = self.spec, self.inp, self.shards, self.spec.rows
        live = int(R - self.classes["masked"])
        nonzero = int(R - self.classes["zero_grad_rows"])
        m = 1 if inp.mask is not None else 0
        o = 4 if self.old is not None else 0
        r = 4 if self.ref is not None else 0
        fwd_logits = live * spec.V * spec.elem_size
        stats = fwd_logits + S * (R * (m + 16) + live * 8)
        combine = R * (m + 21 + 4) + live * (S * 16 + 8 + o + r)
        bwd = per["grpo_loss_bwd"] + (S - 1) * (R * m + live * (4 + o + r + 4) + nonzero * 12) + S * nonzero * 4
        self.classes["vocab_shards"] = S
        self.classes["vocab_starts"] = self.starts
        return {"grpo_vocab_shard_stats": int(stats), "grpo_vocab_combine": int(combine),
                "grpo_loss_bwd_vocab_shard": int(bwd)}

    def e2e_part(self, d, part):
        spec = self.spec
        x, dlog = d["logits"], self._cut(self.dlogits, "bl", part)
        idx, adv, mask, dloss, old, ref = d["idx"], d["adv"], d.get("mask"), d["dloss"], d.get("old"), d.get("ref")
        sl = lambda t, k: t[..., self.starts[k]:self.starts[k + 1]]
        stats = torch.stack([rp.grpo_vocab_shard_stats(sl(x, k), self.starts[k], T=spec.T, idx=idx, mask=mask)
                             for k in range(self.shards)])
        f = rp.grpo_vocab_combine(stats, self.starts, x.shape[0], x.shape[1], T=spec.T, idx=idx, adv=adv, grpo=True,
                                  beta=spec.beta, eps_low=spec.eps_low, eps_high=spec.eps_high, old_logp=old,
                                  ref_logp=ref, mask=mask)
        for k in range(self.shards):
            rp.grpo_loss_bwd_vocab_shard(sl(x, k), self.starts[k], spec.V, idx, adv, dloss, f["logp"], f["lse"],
                                         f["p_rest"], T=spec.T, beta=spec.beta, eps_low=spec.eps_low,
                                         eps_high=spec.eps_high, old_logp=old, ref_logp=ref, mask=mask,
                                         dlogits=sl(dlog, k))
        return {"dlogits": dlog, "loss": f["loss"]}


class EntropySlsmStep(PipelinedE2E):
    """entropy_from_logits, selective_log_softmax_fwd, selective_log_softmax_bwd."""

    oracle_kind = "slsm"

    def __init__(self, spec, seed, device):
        self.spec = spec
        lib = rp.load_library()
        inp = W.generate(spec, seed, device=device)
        self.inp = inp
        R = spec.rows
        f32 = dict(dtype=torch.float32, device=device)
        self.H, self.logp, self.lse = torch.empty(R, **f32), torch.empty(R, **f32), torch.empty(R, **f32)
        self.dlogits = torch.empty(inp.logits.shape, dtype=inp.logits.dtype, device=device)
        self.x_desc, self.dx_desc = rp.rows_of(inp.logits), rp.rows_of(self.dlogits)
        self.stream = torch.cuda.current_stream(device).cuda_stream
        T = spec.T
        self._e, self._f, self._b = lib.entropy_from_logits, lib.selective_log_softmax_fwd, lib.selective_log_softmax_bwd
        self.e_args = (ctypes.byref(self.x_desc), T, _p(self.H), None, self.stream)
        self.f_args = (ctypes.byref(self.x_desc), _p(inp.idx), T, _p(self.logp), _p(self.lse), None, self.stream)
        self.b_args = (ctypes.byref(self.x_desc), _p(inp.idx), _p(inp.upstream), _p(self.lse), T,
                       ctypes.byref(self.dx_desc), None, self.stream)
        self.kernels = [("entropy_from_logits", lambda: self._call(self._e, self.e_args)),
                        ("selective_log_softmax_fwd", lambda: self._call(self._f, self.f_args)),
                        ("selective_log_softmax_bwd", lambda: self._call(self._b, self.b_args))]

    @staticmethod
    def _call(fn, args):
        st = fn(*args)
        if st:
            raise rp.GrpoError(fn.__name__, st)

    def account(self):
        spec = self.spec
        R, V, s = spec.rows, spec.V, spec.elem_size
        self.classes = {"rows": R, "zero_grad_rows": 0, "strided": spec.strided}
        return {k: R * f(V, s) for k, f in SLSM_ROW_BYTES.items()}

    def e2e_inputs(self):
        inp = self.inp
        return {"logits": (inp.logits, "bl"), "idx": (inp.idx, "r"), "up": (inp.upstream, "r")}

    def e2e_outputs(self):
        R = self.spec.rows
        f32 = lambda: ((R,), torch.float32, "r")
        return {"dlogits": (tuple(self.dlogits.shape), self.dlogits.dtype, "bl"), "entropy": f32(), "logp": f32(),
                "lse": f32()}

    def e2e_part(self, d, part):
        T = self.spec.T
        H = rp.entropy_from_logits(d["logits"], T=T)
        lp, lse = rp.selective_log_softmax_fwd(d["logits"], d["idx"], T=T)
        dl = rp.selective_log_softmax_bwd(d["logits"], d["idx"], d["up"], lse, T=T,
                                          dlogits=self._cut(self.dlogits, "bl", part))
        return {"dlogits": dl, "entropy": H, "logp": lp, "lse": lse}


class SeqStep(GrpoStep):
    """Sequence-level GRPO: selective_log_softmax_fwd (logp, lse), grpo_seq_terms (the
    per-sequence ratio, clip and KL terms and the per-token dlogp), then
    selective_log_softmax_bwd (dlogits; rows whose dlogp is 0 are written without a read)."""

    E2E_PART_BYTES = 32 << 20  # public Python API calls per part

    oracle_kind = "seq"
    E2E_WHOLE_SEQUENCES = True

    def __init__(self, spec, seed, device, inputs=None):
        super().__init__(spec, seed, device, inputs)
        lib = rp.load_library()
        inp, o, R, B = self.inp, self.out, spec.rows, spec.B
        f32 = dict(dtype=torch.float32, device=device)
        self.dlogp = torch.empty(R, **f32)
        self.seq_ratio = torch.empty(B, **f32)
        self.seq_clip = torch.empty(B, dtype=torch.uint8, device=device)
        T = spec.T
        self._sf, self._sq, self._sb = (lib.selective_log_softmax_fwd, lib.grpo_seq_terms,
                                        lib.selective_log_softmax_bwd)
        self.sf_args = (ctypes.byref(self.x_desc), _p(inp.idx), T, _p(o["logp"]), _p(o["lse"]), None, self.stream)
        self.sq_args = (B, spec.L, _p(o["logp"]), _p(self.old), _p(self.ref), _p(inp.adv), _p(inp.mask),
                        _p(inp.dloss), spec.beta, spec.eps_low, spec.eps_high, _p(o["loss"]), _p(o["kl"]),
                        _p(self.dlogp), _p(self.seq_ratio), _p(self.seq_clip), self.stream)
        self.sb_args = (ctypes.byref(self.x_desc), _p(inp.idx), _p(self.dlogp), _p(o["lse"]), T,
                        ctypes.byref(self.dx_desc), None, self.stream)
        self.kernels = [("selective_log_softmax_fwd", lambda: self._call(self._sf, self.sf_args)),
                        ("grpo_seq_terms", lambda: self._call(self._sq, self.sq_args)),
                        ("selective_log_softmax_bwd", lambda: self._call(self._sb, self.sb_args))]

    @staticmethod
    def _call(fn, args):
        st = fn(*args)
        if st:
            raise rp.GrpoError(fn.__name__, st)

    def account(self):
        """Minimal bytes.  Forward: every row reads its V logits and idx, writes logp and
        lse.  Sequence terms: every row reads its mask byte and writes loss, kl, dlogp; an
        unmasked row reads logp, old, ref, dloss; every sequence reads A and writes its
        ratio and clip flag.  Backward: every row reads dlogp and writes V dlogits; a row
        whose dlogp is non-zero also reads idx, lse and its V logits."""
        spec, inp = self.spec, self.inp
        R, V, s = spec.rows, spec.V, spec.elem_size
        live = np.ones(R, bool) if inp.mask is None else inp.mask.bool().cpu().numpy()
        zero = (self.dlogp == 0).cpu().numpy()
        m = 1 if inp.mask is not None else 0
        o = 4 if self.old is not None else 0
        r = 4 if self.ref is not None else 0
        n_live, n_zero = int(live.sum()), int(zero.sum())
        self.classes = {"rows": R, "masked": R - n_live, "zero_grad_rows": n_zero,
                        "zero_grad_frac": round(n_zero / R, 4), "seq_level": True,
                        "seq_clipped": int(self.seq_clip.sum())}
        return {"selective_log_softmax_fwd": R * (V * s + 16),
                "grpo_seq_terms": R * (m + 12) + n_live * (8 + o + r) + spec.B * 9,
                "selective_log_softmax_bwd": R * (4 + V * s) + (R - n_zero) * (12 + V * s)}

    def e2e_part(self, d, part):
        spec = self.spec
        b0, b1, l0, l1 = part
        assert (l0, l1) == (0, spec.L), "the sequence-level terms need whole sequences"
        lp, lse = rp.selective_log_softmax_fwd(d["logits"], d["idx"], T=spec.T)
        t = rp.grpo_seq_terms(lp, d["adv"], d["dloss"], B=b1 - b0, L=spec.L, beta=spec.beta, eps_low=spec.eps_low,
                              eps_high=spec.eps_high, old_logp=d.get("old"), ref_logp=d.get("ref"), mask=d.get("mask"))
        dl = rp.selective_log_softmax_bwd(d["logits"], d["idx"], t["dlogp"], lse, T=spec.T,
                                          dlogits=self._cut(self.dlogits, "bl", part))
        return {"dlogits": dl, "loss": t["loss"]}


class EntropyBwdStep(EntropySlsmStep):
    """entropy_from_logits (entropy and lse) then entropy_from_logits_bwd, the gradient of
    sum_r u_r H_r with the workload's upstream gradient u."""

    oracle_kind = "entropy_bwd"

    def __init__(self, spec, seed, device):
        super().__init__(spec, seed, device)
        lib = rp.load_library()
        inp, T = self.inp, spec.T
        self._eb = lib.entropy_from_logits_bwd
        self.e_args = (ctypes.byref(self.x_desc), T, _p(self.H), _p(self.lse), self.stream)
        self.eb_args = (ctypes.byref(self.x_desc), _p(inp.upstream), _p(self.lse), _p(self.H), T,
                        ctypes.byref(self.dx_desc), self.stream)
        self.kernels = [("entropy_from_logits", lambda: self._call(self._e, self.e_args)),
                        ("entropy_from_logits_bwd", lambda: self._call(self._eb, self.eb_args))]

    def account(self):
        """Minimal bytes.  Forward: every row reads its V logits, writes entropy and lse.
        Backward: every row reads u and writes V dlogits; a row with u != 0 also reads
        lse, entropy and its V logits."""
        spec, inp = self.spec, self.inp
        R, V, s = spec.rows, spec.V, spec.elem_size
        n_zero = int((inp.upstream == 0).sum())
        self.classes = {"rows": R, "zero_grad_rows": n_zero, "strided": spec.strided, "entropy_bwd": True}
        return {"entropy_from_logits": R * (V * s + 8),
                "entropy_from_logits_bwd": R * (4 + V * s) + (R - n_zero) * (8 + V * s)}

    def e2e_inputs(self):
        return {"logits": (self.inp.logits, "bl"), "up": (self.inp.upstream, "r")}

    def e2e_outputs(self):
        return {"dlogits": (tuple(self.dlogits.shape), self.dlogits.dtype, "bl"),
                "entropy": ((self.spec.rows,), torch.float32, "r")}

    def e2e_part(self, d, part):
        T = self.spec.T
        H, lse = rp.entropy_from_logits(d["logits"], T=T, return_lse=True)
        dl = rp.entropy_from_logits_bwd(d["logits"], d["up"], lse, H, T=T,
                                        dlogits=self._cut(self.dlogits, "bl", part))
        return {"dlogits": dl, "entropy": H}


def make_spec(args):
    over = {}
    if args.beta is not None:
        over["beta"] = args.beta
    if args.zero_seqs is not None:
        over["zero_adv_seqs"] = args.zero_seqs
    if args.strided:
        over["strided"] = True
    if args.batch is not None:
        over["B"] = args.batch
    return W.get(args.workload, **over)


def step_kind(args, spec):
    """Which pass a bench run times: "grpo", "slsm", "seq" or "entropy_bwd"."""
    if spec.name.startswith("entropy_slsm"):
        return "entropy_bwd" if args.entropy_bwd else "slsm"
    return "seq" if args.seq_level else "grpo"


def make_step(spec, seed, device, fused=False, vocab_shards=0, seq_level=False, entropy_bwd=False):
    if spec.name.startswith("entropy_slsm"):
        return EntropyBwdStep(spec, seed, device) if entropy_bwd else EntropySlsmStep(spec, seed, device)
    if vocab_shards:
        return VocabShardStep(spec, seed, device, vocab_shards)
    if seq_level:
        return SeqStep(spec, seed, device)
    return FusedStep(spec, seed, device) if fused else GrpoStep(spec, seed, device)


# ---------------------------------------------------------------------------
# timing
# ---------------------------------------------------------------------------

def timed_run(step, K, Wm, flush_buf, world, per_kernel=True):
    """Warm up, then time exactly K steps (L2 flushed before each step, outside the
    events).  per_kernel: CUDA events around every kernel, returns per-kernel times [K]
    in ms; else events at the step's start and end only (nothing between the kernels, so
    consecutive kernels overlap their launch with the previous kernel's drain as they do
    in use), returns {"step": [K]}.  Also returns the wall time of the barrier-bracketed
    region."""
    names = [n for n, _ in step.kernels]
    for i in range(Wm):
        flush_buf(i)
        for _, fn in step.kernels:
            fn()
    torch.cuda.synchronize()
    nk = len(step.kernels) if per_kernel else 1
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(K)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(K):
        flush_buf(i + 1)
        e = ev[i]
        e[0].record()
        for k, (_, fn) in enumerate(step.kernels):
            fn()
            if per_kernel:
                e[k + 1].record()
        if not per_kernel:
            e[1].record()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - t0
    if not per_kernel:
        return {"step": [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]}, wall
    per = {n: [ev[i][k].elapsed_time(ev[i][k + 1]) for i in range(K)] for k, n in enumerate(names)}
    return per, wall


def aggregate_max_ms(local_ms: float, world: int, device) -> float:
    """The timed region's length for the whole job: the maximum over ranks."""
    if world <= 1:
        return float(local_ms)
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rates(step_bytes: int, rows: int, K: int, world: int, total_ms: float):
    """(GB/s, rows/s) of the whole job: every rank processed K steps of its own batch of
    the same size, in at most total_ms."""
    sec = total_ms * 1e-3
    return step_bytes * K * world / sec / 1e9, rows * K * world / sec


def e2e_run(step, K, Wm):
    step.e2e_setup()
    for _ in range(max(1, Wm)):
        step.e2e_step()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(K):
        step.e2e_step()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) / K


def entropy_run(step, K, Wm, flush_buf, peak):
    """entropy_from_logits alone over the step's logits (the row pass's entropy kernel,
    reading each row once): Wm untimed launches, then K launches with L2 flushed before
    each and CUDA events around each, on the launching stream."""
    lib = rp.load_library()
    spec = step.spec
    R = spec.rows
    ent = torch.empty(R, dtype=torch.float32, device=step.inp.idx.device)
    args = (ctypes.byref(step.x_desc), spec.T, _p(ent), None, step.stream)

    def call():
        st = lib.entropy_from_logits(*args)
        if st:
            raise rp.GrpoError("entropy_from_logits", st)

    for i in range(Wm):
        flush_buf(i)
        call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        flush_buf(i + 1)
        ev[i][0].record()
        call()
        ev[i][1].record()
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    nbytes = R * SLSM_ROW_BYTES["entropy_from_logits"](spec.V, spec.elem_size)
    gbs = nbytes / (ms * 1e-3) / 1e9
    traffic = measured_traffic("entropy_from_logits", spec)
    return {"kernel": "entropy_from_logits", "value": round(gbs, 2), "unit": "GB/s", "ms": round(ms, 5),
            "bytes": int(nbytes), "rows_per_s": round(R / (ms * 1e-3), 1), "hbm_frac": round(gbs / peak, 4),
            "launches": K, "traffic": traffic,
            "dram_frac": None if traffic is None else round(traffic / (ms * 1e-3) / 1e9 / peak, 4)}


def fused_run(step, K, Wm, flush_buf, peak, step_ms):
    """grpo_loss_fused over the same batch as the fwd + bwd step (the same inputs, dloss
    known in advance, outputs and dlogits into the step's own buffers): Wm untimed
    launches, then K launches with L2 flushed before each and CUDA events around each, on
    the launching stream.  `vs_fwd_bwd_rows` is the step's time over this kernel's, i.e.
    its rows/s over the fwd + bwd step's."""
    lib = rp.load_library()
    spec, inp, o = step.spec, step.inp, step.out
    R = spec.rows
    args = (ctypes.byref(step.x_desc), _p(inp.idx), _p(step.old), _p(step.ref), _p(inp.adv), _p(inp.mask),
            _p(inp.dloss), spec.T, spec.beta, spec.eps_low, spec.eps_high, _p(o["loss"]), _p(o["logp"]),
            _p(o["lse"]), _p(o["kl"]), _p(o["is_clipped"]), _p(o["entropy"]), ctypes.byref(step.dx_desc), None,
            step.stream)

    def call():
        st = lib.grpo_loss_fused(*args)
        if st:
            raise rp.GrpoError("grpo_loss_fused", st)

    for i in range(Wm):
        flush_buf(i)
        call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        flush_buf(i + 1)
        ev[i][0].record()
        call()
        ev[i][1].record()
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    live = np.ones(R, bool) if inp.mask is None else inp.mask.bool().cpu().numpy()
    nbytes = int(fused_row_bytes(spec, live, inp.mask is not None, step.old is not None, step.ref is not None).sum())
    gbs = nbytes / (ms * 1e-3) / 1e9
    traffic = measured_traffic("grpo_loss_fused", spec)
    return {"kernel": "grpo_loss_fused", "value": round(gbs, 2), "unit": "GB/s", "ms": round(ms, 5),
            "bytes": nbytes, "rows_per_s": round(R / (ms * 1e-3), 1), "hbm_frac": round(gbs / peak, 4),
            "vs_fwd_bwd_rows": round(step_ms / ms, 4), "launches": K, "traffic": traffic,
            "dram_frac": None if traffic is None else round(traffic / (ms * 1e-3) / 1e9 / peak, 4)}


# ---------------------------------------------------------------------------
# CPU oracle (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(step, rows):
    """Host copies of one sample of the workload's rows, ready for the oracle."""
    import oracle
    spec, inp = step.spec, step.inp
    r = torch.as_tensor(rows, dtype=torch.int64, device=inp.idx.device)
    x = inp.logits[r // spec.L, r % spec.L].cpu()
    xb = oracle.bf16_bits_to_fp64(x.view(torch.int16).numpy().view(np.uint16)) if x.dtype == torch.bfloat16 \
        else x.double().numpy()
    g = lambda t: None if t is None else t[r].double().cpu().numpy()
    smp = {"x": xb, "idx": inp.idx[r].cpu().numpy(), "adv": oracle.per_row(inp.adv.cpu().numpy(), spec.L)[rows],
           "mask": None if inp.mask is None else inp.mask[r].cpu().numpy()}
    if isinstance(step, GrpoStep):
        smp.update(old=g(step.old), ref=g(step.ref), dloss=g(inp.dloss))
    else:
        smp.update(up=g(inp.upstream))
    if step.oracle_kind == "seq":
        smp["adv_seq"] = inp.adv.cpu().double().numpy()[np.asarray(rows)[::spec.L] // spec.L]
    return smp


def oracle_step(spec, smp, kind):
    import oracle
    if kind == "slsm":
        oracle.entropy_from_logits(smp["x"], spec.T)
        oracle.selective_log_softmax(smp["x"], smp["idx"], spec.T)
        d, _ = oracle.selective_log_softmax_bwd(smp["x"], smp["idx"], smp["up"], spec.T)
    elif kind == "entropy_bwd":
        oracle.entropy_from_logits(smp["x"], spec.T)
        d, _ = oracle.entropy_from_logits_bwd(smp["x"], smp["up"], spec.T)
    elif kind == "seq":
        n_seq = len(smp["adv_seq"])
        d, _, _ = oracle.grpo_seq_loss_bwd(smp["x"], smp["idx"], smp["old"], smp["ref"], smp["adv_seq"], smp["mask"],
                                           smp["dloss"], n_seq, spec.L, spec.T, spec.beta, spec.eps_low, spec.eps_high)
    else:
        oracle.grpo_loss_fwd(smp["x"], smp["idx"], smp["old"], smp["ref"], smp["adv"], smp["mask"], spec.T,
                             spec.beta, spec.eps_low, spec.eps_high)
        d, _ = oracle.grpo_loss_bwd(smp["x"], smp["idx"], smp["old"], smp["ref"], smp["adv"], smp["mask"],
                                    smp["dloss"], spec.T, spec.beta, spec.eps_low, spec.eps_high)
    if spec.dtype == "bf16":
        oracle.round_to_bf16_bits(d)
    else:
        oracle.round_to_fp32(d)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


ORACLE_ROWS = 2048  # rows of the fixed oracle sample
# The workers' first runs over a sample are slower (1.8, 1.4, 1.2 s on 16 Grace cores for
# the 2048 rows at V = 151936), so the cpu_baseline leg takes as many warm-up runs as the
# default reference arm before its median.
ORACLE_WARMUP, ORACLE_REPEATS = 5, 7


def oracle_slice(spec, kind, n=ORACLE_ROWS, seed=11):
    """The fixed seeded slice of rows the oracle is timed on: n consecutive rows starting at
    a seeded multiple of n, or for the sequence-level pass (its ratio is a sum over a
    sequence) the whole sequences of about n rows starting at a seeded sequence."""
    R, L = spec.rows, spec.L
    rng = np.random.default_rng(seed)
    if kind == "seq":
        nseq = max(1, min(spec.B, -(-n // L)))
        b0 = int(rng.integers(0, spec.B // nseq)) * nseq
        return np.arange(b0 * L, (b0 + nseq) * L, dtype=np.int64)
    n = min(n, R)
    r0 = int(rng.integers(0, R // n)) * n
    return np.arange(r0, r0 + n, dtype=np.int64)


def sample_bytes(spec, kind, smp):
    """Minimal bytes of the timed pass over the sample's rows (the same accounting as the
    GPU step's, with the row classes read off the oracle's own results)."""
    import oracle
    n = len(smp["idx"])
    V, s = spec.V, spec.elem_size
    if kind == "entropy_bwd":
        return n * (V * s + 8) + n * (4 + V * s) + int((smp["up"] != 0).sum()) * (8 + V * s)
    if kind == "slsm":
        return n * sum(f(V, s) for f in SLSM_ROW_BYTES.values())
    live = np.ones(n, bool) if smp["mask"] is None else smp["mask"] != 0
    lp, _ = oracle.selective_log_softmax(smp["x"], smp["idx"], spec.T)
    if kind == "seq":
        t = oracle.grpo_seq_terms(lp, smp["old"], smp["ref"], smp["adv_seq"], smp["mask"], smp["dloss"],
                                  n // spec.L, spec.L, spec.beta, spec.eps_low, spec.eps_high)
        m, o, r = (smp["mask"] is not None), 4 * (smp["old"] is not None), 4 * (smp["ref"] is not None)
        nz = int((t["dlogp"] != 0).sum())
        return (n * (V * s + 16) + n * (m + 12) + int(live.sum()) * (8 + o + r) + (n // spec.L) * 9
                + n * (4 + V * s) + nz * (12 + V * s))
    g = oracle.grpo_dlogp(lp, smp["old"], smp["ref"], smp["adv"], smp["mask"], spec.beta, spec.eps_low,
                          spec.eps_high) * smp["dloss"]
    f, b = grpo_row_bytes(spec, live, g == 0, smp["mask"] is not None, smp["old"] is not None,
                          smp["ref"] is not None)
    return int(f.sum() + b.sum())


def _oracle_worker(conn, spec, kind):
    """One host core's share of an oracle sample: keep the part it is sent (a dict), run
    oracle_step on it at every "go" and send back the time it took; None ends the worker."""
    import oracle  # noqa: F401  (imported before any timing)
    part = None
    while True:
        msg = conn.recv()
        if msg is None:
            return
        if isinstance(msg, dict):
            part = msg
            conn.send("ready")
            continue
        t = time.perf_counter()
        oracle_step(spec, part, kind)
        conn.send(time.perf_counter() - t)


class OraclePool:
    """The oracle on several host cores: spawned worker processes (one per core, one numpy
    thread each) run oracle_step, unchanged, on disjoint parts of one sample (whole
    sequences for the sequence-level pass).  The parts are handed over once, before any
    clock starts; a run's time is the wall time from the start signal until the last part
    is done."""

    _THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")

    def __init__(self, n, spec, kind):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        saved = {k: os.environ.get(k) for k in self._THREAD_VARS}
        for k in self._THREAD_VARS:
            os.environ[k] = "1"
        self.spec, self.kind, self.conns, self.procs, self.active = spec, kind, [], [], []
        try:
            for _ in range(n):
                a, b = ctx.Pipe()
                p = ctx.Process(target=_oracle_worker, args=(b, spec, kind), daemon=True)
                p.start()
                self.conns.append(a)
                self.procs.append(p)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def split(self, smp):
        """The sample cut into at most len(workers) parts of whole units."""
        unit = self.spec.L if self.kind == "seq" else 1
        units = len(smp["idx"]) // unit
        n = min(len(self.conns), units)
        bounds = [unit * (units * k // n) for k in range(n + 1)]
        parts = []
        for lo, hi in zip(bounds[:-1], bounds[1:]):
            part = {}
            for k, v in smp.items():
                if v is None or np.ndim(v) == 0:
                    part[k] = v
                elif k == "adv_seq":
                    part[k] = v[lo // unit:hi // unit]
                else:
                    part[k] = v[lo:hi]
            parts.append(part)
        return parts

    def load(self, smp):
        """Hand the sample's parts to the workers (untimed)."""
        parts = self.split(smp)
        self.active = self.conns[:len(parts)]
        for c, part in zip(self.active, parts):
            c.send(part)
        for c in self.active:
            assert c.recv() == "ready"

    def go(self):
        """Wall seconds of one run of the loaded sample over the workers."""
        t = time.perf_counter()
        for c in self.active:
            c.send("go")
        for c in self.active:
            c.recv()
        return time.perf_counter() - t

    def close(self):
        for c in self.conns:
            c.send(None)
        for p in self.procs:
            p.join(timeout=30)


def time_oracle(spec, kind, smp, warmup=1, repeats=3):
    """The oracle over one sample on all host cores, timed the one way both the
    cpu_baseline and the reference arm use: the sample handed to the workers, `warmup`
    untimed runs, then `repeats` timed runs.  Returns (median seconds, cores used, times)."""
    cores = host_cores()
    if cores <= 1:
        times = []
        for i in range(warmup + repeats):
            t = time.perf_counter()
            oracle_step(spec, smp, kind)
            times.append(time.perf_counter() - t)
        return statistics.median(times[warmup:]), 1, times[warmup:]
    pool = OraclePool(cores, spec, kind)
    try:
        pool.load(smp)
        for _ in range(warmup):
            pool.go()
        times = [pool.go() for _ in range(repeats)]
        return statistics.median(times), len(pool.active), times
    finally:
        pool.close()


def one_core_figure(spec, kind, smp, budget_s=8.0):
    """The oracle on this process's one thread over the sample's leading rows (whole
    sequences for the sequence-level pass), as many as fit in about budget_s."""
    unit = spec.L if kind == "seq" else 1
    n = len(smp["idx"])
    cut = lambda k: {key: (v if v is None or np.ndim(v) == 0 else (v[:k // unit] if key == "adv_seq" else v[:k]))
                     for key, v in smp.items()}
    probe = cut(min(n, max(unit, 8)))
    t = time.perf_counter()
    oracle_step(spec, probe, kind)
    per_row = (time.perf_counter() - t) / len(probe["idx"])
    k = max(unit, min(n, int(budget_s / max(per_row, 1e-9)) // unit * unit))
    sub = cut(k)
    t = time.perf_counter()
    oracle_step(spec, sub, kind)
    dt = time.perf_counter() - t
    return {"value": round(sample_bytes(spec, kind, sub) / dt / 1e9, 6), "cores": 1,
            "rows_per_s": round(len(sub["idx"]) / dt, 2), "rows": len(sub["idx"]), "seconds": round(dt, 2)}


def cpu_baseline(step):
    """The oracle, as it stands, on the fixed seeded slice of this workload's rows, on all
    host cores (time_oracle), with a one-core figure beside it."""
    spec, kind = step.spec, step.oracle_kind
    rows = oracle_slice(spec, kind)
    smp = oracle_sample(step, rows)
    nbytes = sample_bytes(spec, kind, smp)
    one = one_core_figure(spec, kind, smp)
    dt, used, times = time_oracle(spec, kind, smp, warmup=ORACLE_WARMUP, repeats=ORACLE_REPEATS)
    return {"value": round(nbytes / dt / 1e9, 6), "unit": "GB/s", "cores": used, "kind": "oracle",
            "rows_per_s": round(len(rows) / dt, 2), "one_core": one,
            "seconds": [round(t, 3) for t in times],
            "sample": f"rows [{rows[0]}, {rows[-1] + 1}) of {spec.rows} of {spec.name} ({kind} fwd+bwd, fp64 "
                      f"numpy), split over {used} spawned processes of one thread each; {ORACLE_WARMUP} warm-up "
                      f"runs, then the median of {len(times)}: {dt:.2f} s"}


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------

def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default: about 2 s of steps)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="sweep_b16_l4096_v151936",
                    choices=list(GRPO_WORKLOADS) + ["entropy_slsm_b16_l4096_v32000", LINEAR_WORKLOAD])
    ap.add_argument("--chunk-rows", type=int, default=2048,
                    help="rows per chunk of the LM-head workload (grpo_fused_linear)")
    ap.add_argument("--beta", type=float, default=None)
    ap.add_argument("--zero-seqs", type=int, default=None)
    ap.add_argument("--strided", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="sequences B instead of the workload's own (a smaller case of the same rows, e.g. for ncu)")
    ap.add_argument("--fused", action="store_true",
                    help="GRPO workloads: time grpo_loss_fused (one kernel) instead of grpo_loss_fwd + grpo_loss_bwd")
    ap.add_argument("--vocab-shards", type=int, default=0,
                    help="GRPO workloads: the vocabulary-parallel step of this many shards, run shard after shard")
    ap.add_argument("--seq-level", action="store_true",
                    help="GRPO workloads: the sequence-level step (selective_log_softmax_fwd, grpo_seq_terms, "
                         "selective_log_softmax_bwd)")
    ap.add_argument("--entropy-bwd", action="store_true",
                    help="entropy_slsm workload: entropy_from_logits (with lse) then entropy_from_logits_bwd")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args(argv)


def base_line(args, spec, world):
    return {"metric": METRIC, "unit": "GB/s", "n_gpus": world, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "data": "synthetic",
            "config": {"workload": spec.name, "pass": step_kind(args, spec), "B": spec.B, "L": spec.L, "V": spec.V,
                       "T": spec.T,
                       "beta": spec.beta, "eps_low": spec.eps_low, "eps_high": spec.eps_high,
                       "logits_dtype": spec.dtype, "strided": spec.strided,
                       "l2": "flushed before every timed step (256 MB write + 256 MB read, not timed)",
                       "parallelism": f"{world} independent batch(es), one per GPU"}}


def run_reference(args):
    """The oracle as the reference arm, on the host cores only: inputs drawn on the CPU
    from the same generators (only the sampled rows' logits), old/ref placed with the
    oracle's own logp, and each step one run of the fixed seeded slice of the workload's
    rows (fwd + bwd), timed as cpu_baseline times it."""
    rank, world, local = dist_env()
    if rank != 0:
        return 0
    import oracle  # the one other place bench.py runs the oracle
    if args.workload == LINEAR_WORKLOAD:
        return run_reference_linear(args, oracle)
    spec = make_spec(args)
    kind = step_kind(args, spec)
    inp = W.generate(spec, args.seed, device="cpu", with_logits=False)
    L = spec.L
    grpo = kind in ("grpo", "seq")
    rows = oracle_slice(spec, kind)
    x = W.logits_rows(spec, args.seed, int(rows[0]), int(rows[-1]) + 1)
    xd = oracle.bf16_bits_to_fp64(x.view(torch.int16).numpy().view(np.uint16)) if x.dtype == torch.bfloat16 \
        else x.double().numpy()
    del x
    smp = {"x": xd, "idx": inp.idx.numpy()[rows], "adv": oracle.per_row(inp.adv.numpy(), L)[rows],
           "mask": None if inp.mask is None else inp.mask.numpy()[rows]}
    if grpo:
        lp, _ = oracle.selective_log_softmax(xd, smp["idx"], spec.T)
        add = lambda off: None if off is None else oracle.round_to_fp32(lp + off.numpy()[rows]).astype(np.float64)
        smp["old"] = add(inp.old_offset)
        smp["ref"] = add(inp.ref_offset) if spec.beta != 0 else None
        smp["dloss"] = inp.dloss.numpy().astype(np.float64)[rows]
    else:
        smp["up"] = inp.upstream.numpy().astype(np.float64)[rows]
    if kind == "seq":
        smp["adv_seq"] = inp.adv.numpy().astype(np.float64)[rows[::L] // L]

    K = args.steps if args.steps is not None else 10
    Wm = args.warmup
    nbytes = sample_bytes(spec, kind, smp)
    med, used, times = time_oracle(spec, kind, smp, warmup=max(1, Wm), repeats=max(1, K))
    value = nbytes / med / 1e9
    line = base_line(args, spec, 1)
    line.update({"impl": "reference", "value": round(value, 6), "steps": K, "warmup": Wm,
                 "ms_per_step": round(1e3 * med, 3), "dtype": "f64",
                 "rows_per_s": round(len(rows) / med, 2)})
    sample_txt = (f"rows [{rows[0]}, {rows[-1] + 1}) of {spec.rows} of {spec.name} per step ({kind} fwd+bwd, "
                  f"fp64 numpy), split over {used} spawned processes of one thread each; the median of "
                  f"{len(times)} steps after {max(1, Wm)} warm-up")
    line["cpu_baseline"] = {"value": line["value"], "unit": "GB/s", "cores": used, "kind": "oracle",
                            "sample": sample_txt}
    line["e2e"] = {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    print(json.dumps(line), flush=True)
    return 0


def run_reference_linear(args, oracle):
    """The oracle's fused_linear_grpo as the reference arm of the LM-head workload: each
    step a bounded sample of rows against the whole head weight, on the host."""
    spec = W.get(LINEAR_WORKLOAD)
    li = W.generate_linear(spec, args.seed, device="cpu")
    Wf = oracle.bf16_bits_to_fp64(li.weight.view(torch.int16).numpy().view(np.uint16))
    adv_rows = oracle.per_row(li.adv.numpy(), spec.L)

    def step(rows):
        hf = oracle.bf16_bits_to_fp64(li.hidden[rows].view(torch.int16).numpy().view(np.uint16))
        lp, _ = oracle.selective_log_softmax(hf @ Wf.T, li.idx.numpy()[rows], spec.T)
        old = oracle.round_to_fp32(lp + li.old_offset.numpy()[rows]).astype(np.float64)
        ref = oracle.round_to_fp32(lp + li.ref_offset.numpy()[rows]).astype(np.float64)
        mask = None if li.mask is None else li.mask.numpy()[rows]
        t = time.perf_counter()
        oracle.fused_linear_grpo(hf, Wf, li.idx.numpy()[rows], old, ref, adv_rows[rows], mask,
                                 li.dloss.numpy().astype(np.float64)[rows], spec.T, spec.beta, spec.eps_low,
                                 spec.eps_high)
        return time.perf_counter() - t

    K = args.steps if args.steps is not None else 10
    Wm = args.warmup
    per_row = step(W.sample_rows(spec.rows, 4, 3)) / 4
    n = int(max(1, min(spec.rows, 150.0 / max(1, K + Wm) / max(per_row, 1e-9))))
    times = [step(W.sample_rows(spec.rows, n, 100 + i)) for i in range(Wm + K)][Wm:]
    total = sum(times)
    value = n * K / total
    line = {"metric": LINEAR_METRIC, "unit": "rows/s", "n_gpus": 1, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "data": "synthetic", "impl": "reference",
            "config": {"workload": spec.name, "B": spec.B, "L": spec.L, "H": spec.H, "V": spec.V},
            "value": round(value, 4), "steps": K, "warmup": Wm, "ms_per_step": round(1e3 * total / K, 3),
            "dtype": "f64", "rows_per_s": round(value, 4)}
    line["cpu_baseline"] = {"value": line["value"], "unit": "rows/s", "cores": torch.get_num_threads(),
                            "kind": "oracle",
                            "sample": f"{n} of {spec.rows} rows per step (fp64 numpy, the full head weight)"}
    line["e2e"] = {"value": line["value"], "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == LINEAR_WORKLOAD:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py needs a CUDA GPU: the row pass has no CPU path")
        return run_linear(args)
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU: the row pass has no CPU path")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
    spec = make_spec(args)
    step = make_step(spec, args.seed + rank, device, fused=args.fused, vocab_shards=args.vocab_shards,
                     seq_level=args.seq_level, entropy_bwd=args.entropy_bwd)
    flush_buf = L2Flush(device)

    # one untimed step to classify rows, then calibrate the step count
    for _, fn in step.kernels:
        fn()
    torch.cuda.synchronize()
    per_launch = step.account()
    step_bytes = sum(per_launch.values())
    if args.steps is None:
        probe, _ = timed_run(step, 5, 1, flush_buf, 1)
        step_ms = sum(statistics.mean(v) for v in probe.values()) + 0.05
        K = int(min(20000, max(20, math.ceil(2000.0 / step_ms))))
    else:
        K = args.steps
    Wm = max(3, args.warmup)

    # the headline: events at step boundaries only; then a second timed pass with events
    # around every kernel for the per-kernel table and the roofline
    clocks = ClockSampler(local)
    clocks.start()
    steps, wall = timed_run(step, K, Wm, flush_buf, world, per_kernel=False)
    per, _ = timed_run(step, K, Wm, flush_buf, world, per_kernel=True)
    clk = clocks.stop()

    kern_ms = {n: statistics.mean(v) for n, v in per.items()}
    step_ms = statistics.mean(steps["step"])
    total_ms = aggregate_max_ms(sum(steps["step"]), world, device)
    value, rows_per_s = whole_job_rates(step_bytes, spec.rows, K, world, total_ms)

    peak, peak_src = load_peaks()
    dom = max(kern_ms, key=kern_ms.get)
    achieved = per_launch[dom] / (kern_ms[dom] * 1e-3) / 1e9
    traffic = measured_traffic(dom, spec)

    e2e = None
    if not args.no_e2e:
        Ke = min(K, max(5, int(1500.0 / max(step_ms, 1e-3) / 10)), 200)
        if world > 1:  # every rank times the same number of steps
            Ke = int(aggregate_max_ms(float(Ke), world, device))
        ms = aggregate_max_ms(e2e_run(step, Ke, 2), world, device)  # the slowest rank's time per step
        e2e_val = step_bytes * world / (ms * 1e-3) / 1e9
        e2e = {"value": round(e2e_val, 3), "unit": "GB/s", "h2d_bytes_per_step": int(step.h2d),
               "d2h_bytes_per_step": int(step.d2h), "ms_per_step": round(ms, 4), "steps": Ke,
               "parts": len(step.e2e_bounds), "outputs_copied_back": step.e2e_outputs_kept,
               "path": ("the C-ABI entry points with outputs allocated once" if not step.E2E_VIEWS else
                        "the public Python API") +
                       ", pinned host inputs, outputs copied back; the batch in parts (whole sequences, or token "
                       "ranges of one sequence for the token-level passes), the logits copied in, the kernels and "
                       "the outputs copied out per part on three streams"}

    ent = fus = None
    if step_kind(args, spec) == "grpo" and not args.vocab_shards:
        ent = entropy_run(step, K, Wm, flush_buf, peak)
        if not args.fused:  # the same batch through the single-read kernel, beside the fwd + bwd step
            fus = fused_run(step, K, Wm, flush_buf, peak, step_ms)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(step)

    if rank == 0:
        line = base_line(args, spec, world)
        line["config"].update(step.classes)
        line.update({
            "value": round(value, 2), "steps": K, "warmup": Wm, "ms_per_step": round(step_ms, 5),
            "dtype": spec.dtype, "rows_per_s": round(rows_per_s, 1),
            "hbm_frac": round(value / world / peak, 4),
            "bytes_per_step": int(step_bytes),
            "kernels": {n: {"ms": round(kern_ms[n], 5), "bytes": int(per_launch[n]),
                            "GB_per_s": round(per_launch[n] / (kern_ms[n] * 1e-3) / 1e9, 1)} for n in kern_ms},
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                         "dram_frac": None if traffic is None else
                         round(traffic / (kern_ms[dom] * 1e-3) / 1e9 / peak, 4),
                         "source_hash": kernel_source_hash(dom) if dom in KERNEL_UNITS else None,
                         "peak_source": peak_src,
                         "algorithmic_bytes_per_launch": int(per_launch[dom])},
            "cpu_baseline": cpu, "e2e": e2e, "entropy": ent, "fused": fus,
            "gpu_launches": getattr(step, "launches_per_step", len(step.kernels)) * K,
            "gpu_launches_note": "in the headline pass (the per-kernel pass launches as many again)",
            "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"],
                       "samples": clk["samples"]},
            "timed_wall_s": round(wall, 3), "kernel_source": kernel_source_hash(),
            "timing": {"value": "CUDA events at the start and end of each step, none between its kernels",
                       "kernels": "a second pass of the same K steps with CUDA events around every kernel",
                       "kernels_sum_ms": round(sum(kern_ms.values()), 5)},
        })
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
