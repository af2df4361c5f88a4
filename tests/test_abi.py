"""The C ABI on the CPU: the library loads, exports every function the header declares,
and rejects bad arguments on the host before any CUDA call (fake device addresses are
never dereferenced: each case fails validation, or has zero rows, before a launch)."""
import ctypes
import math
import os
import re

import pytest
import torch

from rl_fine_tuning_pass_gb300 import binding
from rl_fine_tuning_pass_gb300.build import ROOT, build

HEADER = os.path.join(ROOT, "include", "grpo_rowpass.h")
FAKE = 0x7F0000100000          # 16-byte aligned, never dereferenced
P = ctypes.c_void_p


@pytest.fixture(scope="module")
def lib():
    build()
    return binding.load_library()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


def test_header_functions_are_exported(lib):
    names = header_functions()
    assert set(names) == set(binding.EXPORTED), names
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"


def test_status_strings(lib):
    for code in range(4):
        s = binding.status_string(code)
        assert s.startswith("GRPO_")
    assert "unknown" in binding.status_string(99)


def rows(ptr=FAKE, dtype=binding.GRPO_BF16, B=2, L=3, V=64, sb=None, sl=None, reserved=0):
    sl = V if sl is None else sl
    sb = L * sl if sb is None else sb
    return binding.GrpoRows(ptr, dtype, reserved, B, L, V, sb, sl)


def fwd(lib, x, T=1.0, beta=0.0, el=0.2, eh=0.2, idx=FAKE, adv=FAKE, ref=None, outs=FAKE):
    return lib.grpo_loss_fwd(ctypes.byref(x), idx, None, ref, adv, None, T, beta, el, eh,
                             outs, outs + 64, outs + 128, None, None, None, None, None)


def bwd(lib, x, dx, T=1.0, beta=0.0):
    return lib.grpo_loss_bwd(ctypes.byref(x), FAKE, None, None, FAKE, None, FAKE, FAKE, FAKE,
                             T, beta, 0.2, 0.2, ctypes.byref(dx), None, None)


INV, UNS = binding.GRPO_ERR_INVALID_ARG, binding.GRPO_ERR_UNSUPPORTED


@pytest.mark.parametrize("case,want", [
    (dict(ptr=None), INV), (dict(dtype=7), INV), (dict(reserved=1), INV), (dict(V=0), INV),
    (dict(B=-1), INV), (dict(sl=-64), INV), (dict(ptr=FAKE + 1), INV),
    (dict(V=(1 << 30) + 1), UNS), (dict(B=1 << 16, L=1 << 15), UNS),
])
def test_bad_logits_rejected(lib, case, want):
    assert fwd(lib, rows(**case)) == want


@pytest.mark.parametrize("kw", [dict(T=0.0), dict(T=-1.0), dict(T=math.inf), dict(T=math.nan),
                                dict(beta=-0.1), dict(beta=math.nan), dict(el=1.5), dict(el=-0.1),
                                dict(eh=math.inf), dict(idx=None), dict(idx=FAKE + 4), dict(adv=None),
                                dict(beta=0.04, ref=None), dict(outs=FAKE + 2)])
def test_bad_scalars_and_pointers_rejected(lib, kw):
    assert fwd(lib, rows(), **kw) == INV


def test_zero_rows_is_a_no_op(lib):
    assert fwd(lib, rows(B=0)) == binding.GRPO_OK
    assert fwd(lib, rows(ptr=None, B=0), idx=None, adv=None, outs=0) == binding.GRPO_OK
    assert fwd(lib, rows(L=0)) == binding.GRPO_OK
    x0 = rows(B=0)
    assert lib.entropy_from_logits(ctypes.byref(x0), 1.0, FAKE, None, None) == binding.GRPO_OK


def test_dlogits_validation(lib):
    x = rows()
    # partial overlap with the logits
    assert bwd(lib, x, rows(ptr=FAKE + 128)) == INV
    # dtype / shape mismatch
    assert bwd(lib, x, rows(ptr=FAKE + (1 << 20), dtype=binding.GRPO_FP32)) == INV
    assert bwd(lib, x, rows(ptr=FAKE + (1 << 20), V=32)) == INV
    # overlapping output rows
    assert bwd(lib, x, rows(ptr=FAKE + (1 << 20), sl=16)) == INV
    # zero rows with valid descriptors: accepted, nothing launched
    assert bwd(lib, rows(B=0), rows(B=0, ptr=FAKE + (1 << 20))) == binding.GRPO_OK
    assert bwd(lib, rows(L=0), rows(L=0)) == binding.GRPO_OK  # exact alias, no rows
    assert bwd(lib, x, rows(ptr=FAKE + (1 << 20)), T=0.0) == INV


def test_fused_validation(lib):
    x = rows()
    def fused(dx, T=1.0, dloss=FAKE, beta=0.0, ref=None):
        return lib.grpo_loss_fused(ctypes.byref(x), FAKE, None, ref, FAKE, None, dloss, T, beta, 0.2, 0.2,
                                   FAKE, FAKE + 64, FAKE + 128, None, None, None, ctypes.byref(dx), None, None)
    far = rows(ptr=FAKE + (1 << 20))
    assert fused(rows(ptr=FAKE + 128)) == INV          # partial overlap with the logits
    assert fused(far, dloss=None) == INV               # dloss required
    assert fused(far, T=0.0) == INV
    assert fused(far, beta=0.1) == INV                 # ref_logp required when beta > 0
    assert fused(rows(ptr=FAKE + (1 << 20), V=32)) == INV
    x0 = rows(B=0)
    assert lib.grpo_loss_fused(ctypes.byref(x0), None, None, None, None, None, None, 1.0, 0.0, 0.2, 0.2,
                               None, None, None, None, None, None, ctypes.byref(rows(B=0, ptr=None)),
                               None, None) == binding.GRPO_OK


def test_seq_terms_validation(lib):
    def seq(B=2, L=3, logp=FAKE, beta=0.0, ref=None, el=0.2, dlogp=FAKE):
        return lib.grpo_seq_terms(B, L, logp, None, ref, FAKE, None, FAKE, beta, el, 0.2, FAKE, None, dlogp,
                                  None, None, None)
    assert seq(B=-1) == INV
    assert seq(logp=None) == INV
    assert seq(dlogp=None) == INV
    assert seq(beta=0.1) == INV
    assert seq(el=2.0) == INV
    assert seq(logp=FAKE + 2) == INV
    assert seq(B=1 << 16, L=1 << 16) == UNS
    assert seq(B=0, logp=None, dlogp=None) == binding.GRPO_OK


def test_slsm_and_entropy_validation(lib):
    x = rows()
    assert lib.selective_log_softmax_fwd(ctypes.byref(x), None, 1.0, FAKE, FAKE, None, None) == INV
    assert lib.selective_log_softmax_fwd(ctypes.byref(x), FAKE, 0.0, FAKE, FAKE, None, None) == INV
    assert lib.selective_log_softmax_fwd(ctypes.byref(x), FAKE, 1.0, FAKE, FAKE, FAKE + 2, None) == INV
    assert lib.entropy_from_logits(ctypes.byref(x), 1.0, None, None, None) == INV
    assert lib.entropy_from_logits(ctypes.byref(x), math.nan, FAKE, None, None) == INV
    assert lib.entropy_from_logits(ctypes.byref(x), 1.0, FAKE, FAKE + 2, None) == INV
    far = rows(ptr=FAKE + (1 << 20))
    assert lib.entropy_from_logits_bwd(ctypes.byref(x), None, FAKE, FAKE, 1.0, ctypes.byref(far), None) == INV
    assert lib.entropy_from_logits_bwd(ctypes.byref(x), FAKE, FAKE, FAKE, 0.0, ctypes.byref(far), None) == INV
    assert lib.entropy_from_logits_bwd(ctypes.byref(x), FAKE, FAKE, FAKE, 1.0,
                                       ctypes.byref(rows(ptr=FAKE + 64)), None) == INV
    dx = rows(ptr=FAKE + 64)
    assert lib.selective_log_softmax_bwd(ctypes.byref(x), FAKE, FAKE, FAKE, 1.0, ctypes.byref(dx),
                                         None, None) == INV
    assert lib.selective_log_softmax_bwd(ctypes.byref(x), FAKE, None, FAKE, 1.0,
                                         ctypes.byref(rows(ptr=FAKE + (1 << 20))), None, None) == INV


def test_vocab_parallel_validation(lib):
    """The vocabulary-shard entry points reject bad shards, starts and pointer sets on the
    host, before any launch."""
    x = rows()
    def stats(T=1.0, start=0, out=FAKE, idx=None):
        return lib.grpo_vocab_shard_stats(ctypes.byref(x), start, idx, None, T, out, None)
    assert stats(T=0.0) == INV
    assert stats(start=-1) == INV
    assert stats(out=None) == INV
    assert stats(out=FAKE + 8) == INV                  # stats need 16-byte alignment
    assert stats(idx=FAKE + 4) == INV
    assert lib.grpo_vocab_shard_stats(ctypes.byref(rows(B=0)), 0, None, None, 1.0, None, None) == binding.GRPO_OK

    def comb(world=2, starts=(0, 10, 64), idx=FAKE, logp=FAKE + 64, lse=FAKE + 128, loss=None, adv=None,
             st=FAKE, p_rest=None, beta=0.0, ref=None, kl=None):
        arr = (ctypes.c_int64 * len(starts))(*starts)
        return lib.grpo_vocab_combine(world, st, arr, 2, 8, idx, None, ref, adv, None, 1.0, beta, 0.2, 0.2,
                                      loss, logp, lse, kl, None, None, p_rest, None, None)
    assert comb(world=0, starts=(0,)) == INV
    assert comb(world=65, starts=tuple(range(66))) == INV
    assert comb(starts=(1, 10, 64)) == INV                       # must start at 0
    assert comb(starts=(0, 10, 10)) == INV                       # empty shard
    assert comb(starts=(0, 20, 10)) == INV                       # decreasing
    assert comb(st=FAKE + 4) == INV                              # 16-byte stats
    assert comb(idx=None) == INV                                 # logp without idx
    assert comb(idx=None, logp=None, p_rest=FAKE) == INV         # p_rest without idx
    assert comb(lse=None) == INV
    assert comb(loss=FAKE + 192, adv=None) == INV                # GRPO terms need adv
    assert comb(loss=FAKE + 192, adv=FAKE, beta=0.1) == INV      # and ref when beta > 0
    assert comb(kl=FAKE) == INV                                  # kl only with the GRPO terms

    far = rows(ptr=FAKE + (1 << 20))
    def sbwd(start=0, total=64, dx=far, p_rest=FAKE, T=1.0):
        return lib.grpo_loss_bwd_vocab_shard(ctypes.byref(x), start, total, FAKE, None, None, FAKE, None, FAKE,
                                             FAKE, FAKE, p_rest, T, 0.0, 0.2, 0.2, ctypes.byref(dx), None, None)
    assert sbwd(total=63) == INV                                 # shard past the vocabulary
    assert sbwd(start=-1) == INV
    assert sbwd(p_rest=None) == INV
    assert sbwd(T=0.0) == INV
    assert sbwd(dx=rows(ptr=FAKE + 64)) == INV                   # partial overlap
    assert lib.selective_log_softmax_bwd_vocab_shard(ctypes.byref(x), 8, 60, FAKE, FAKE, FAKE, FAKE, 1.0,
                                                     ctypes.byref(far), None, None) == INV


def test_fused_linear_validation(lib):
    """Shapes, alignment and the workspace size are checked on the host before any launch."""
    need = ctypes.c_uint64(0)
    assert lib.grpo_fused_linear_workspace_size(64, 1000, 16, ctypes.byref(need)) == binding.GRPO_OK
    assert need.value >= 1000 * 16 * 2 + 64 * 16 * 2
    assert lib.grpo_fused_linear_workspace_size(64, 0, 16, ctypes.byref(need)) == INV
    assert lib.grpo_fused_linear_workspace_size(64, 1000, 0, ctypes.byref(need)) == INV
    assert lib.grpo_fused_linear_workspace_size(60, 1000, 16, ctypes.byref(need)) == INV   # H % 8 != 0
    assert lib.grpo_fused_linear_workspace_size(64, 1000, 16, ctypes.byref(need)) == binding.GRPO_OK
    big = need.value

    def call(H=64, V=1000, hidden=FAKE, weight=FAKE, ws=FAKE, ws_bytes=big, chunk=16, T=1.0, beta=0.0, ref=None,
             idx=FAKE, gh=None, B=2, L=8):
        return lib.grpo_fused_linear(hidden, weight, B, L, H, V, idx, None, ref, FAKE, None, FAKE, T, beta, 0.2, 0.2,
                                     chunk, ws, ws_bytes, FAKE, FAKE, FAKE, None, None, None, gh, None, None, None)
    assert call(H=60) == INV                       # H must be a multiple of 8
    assert call(hidden=FAKE + 8) == INV             # 16-byte operands
    assert call(weight=None) == INV
    assert call(ws=FAKE + 128) == INV               # 256-byte workspace
    assert call(ws_bytes=big - 1) == INV            # too small for V, chunk
    assert call(chunk=0) == INV
    assert call(T=0.0) == INV
    assert call(beta=0.1) == INV                    # ref_logp required when beta > 0
    assert call(idx=None) == INV
    assert call(gh=FAKE + 4) == INV
    assert call(B=0) == binding.GRPO_OK             # no rows: nothing launched


def test_rows_of_strides():
    import torch
    base = torch.empty(4, 9, 16, dtype=torch.bfloat16)
    v = base[:, :-1, :]
    r = binding.rows_of(v)
    assert (r.B, r.L, r.V, r.stride_b, r.stride_l, r.dtype) == (4, 8, 16, 144, 16, binding.GRPO_BF16)
    r2 = binding.rows_of(torch.empty(5, 7, dtype=torch.float32))
    assert (r2.B, r2.L, r2.V, r2.stride_l) == (1, 5, 7, 7)
    with pytest.raises(ValueError):
        binding.rows_of(torch.empty(4, 8, dtype=torch.float32).t())


def test_autograd_wrappers_have_no_cpu_path():
    """The autograd wrappers marshal into the CUDA library only: CPU tensors are refused
    before any call, never computed some other way."""
    from rl_fine_tuning_pass_gb300 import autograd as ag
    x = torch.randn(2, 3, 8, requires_grad=True)
    idx = torch.zeros(6, dtype=torch.int64)
    with pytest.raises(ValueError, match="CUDA"):
        ag.selective_log_softmax(x, idx)
    with pytest.raises(ValueError, match="CUDA"):
        ag.entropy(x)
    with pytest.raises(ValueError, match="CUDA"):
        ag.grpo_loss(x, idx, torch.zeros(2))


def test_a_failed_launch_returns_grpo_err_cuda():
    """A call whose arguments pass validation but whose launch fails returns
    GRPO_ERR_CUDA and does not crash.  The failure is made on the host: the call runs in a
    child process with no CUDA device visible, so the launch is refused before any kernel
    exists and the fake device addresses are never dereferenced, on any machine."""
    import subprocess
    import sys
    code = (
        "import ctypes, sys\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "from rl_fine_tuning_pass_gb300 import binding\n"
        "lib = binding.load_library()\n"
        f"F = {FAKE}\n"
        "x = binding.GrpoRows(F, binding.GRPO_BF16, 0, 2, 3, 64, 192, 64)\n"
        "st = lib.grpo_loss_fwd(ctypes.byref(x), F, None, None, F, None, 1.0, 0.0, 0.2, 0.2,\n"
        "                       F, F + 64, F + 128, None, None, None, None, None)\n"
        "print(st)\n"
    )
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    build()
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.strip().splitlines()[-1] == str(binding.GRPO_ERR_CUDA)
