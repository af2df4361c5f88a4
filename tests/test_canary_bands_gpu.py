"""Out-of-bounds write checks for every C-ABI entry point (GPU).

compute-sanitizer is not available on the machines these kernels are tested on, so
writes are checked with guard bands: every output array sits inside a larger device
buffer whose every element first holds a NaN bit pattern that no kernel can produce (a
signalling-NaN payload: arithmetic only ever yields quiet NaNs, and the kernels' own NaN
markers are quiet).  After the call:

* every element outside the declared output -- the head before the first row, the gap
  between rows, the tail after the last row, and 64 elements on both sides of each
  per-row array -- must still hold the pattern;
* every element inside it must have been written (no pattern left), including the
  masked rows, the zero rows and the ragged V % 8 tails.

The logits rows start at odd offsets (not 16-byte aligned) and the dlogits rows are out
of phase with them, so the split head / vector body / scalar tail paths of the kernels
are all exercised.  Values are checked by the parity tests; here only where the kernels
write.
"""

import ctypes

import numpy as np
import pytest
import torch

from rl_fine_tuning_pass_gb300 import binding as rp

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]
DEV = "cuda"
BAND = 64  # guard elements on each side of a per-row array
CANARY = {torch.bfloat16: (torch.int16, 0x7FA5), torch.float32: (torch.int32, 0x7FA5A5A5),
          torch.uint8: (torch.uint8, 0xA5)}
VS = [1, 7, 9, 513, 40000, 151936]
HEADS = [1, 3]


@pytest.fixture(scope="module", autouse=True)
def _library():
    from rl_fine_tuning_pass_gb300.build import build
    build()
    rp.load_library()


def _fill(buf):
    it, pat = CANARY[buf.dtype]
    v = pat if it != torch.int32 else np.int32(np.uint32(pat).view(np.int32)).item()
    buf.view(it).fill_(v)


def _is_canary(t):
    it, pat = CANARY[t.dtype]
    v = pat if it != torch.int32 else np.int32(np.uint32(pat).view(np.int32)).item()
    return t.view(it) == v


class Banded:
    """n elements between two guard bands; `t` is the declared array."""

    def __init__(self, n, dtype, zero_inside=False, band=BAND):
        self.n, self.band = n, band
        self.buf = torch.empty(n + 2 * band, dtype=dtype, device=DEV)
        _fill(self.buf)
        self.t = self.buf[band:band + n]
        if zero_inside:
            self.t.zero_()

    @property
    def ptr(self):
        return self.t.data_ptr()

    def check(self, what, written=True):
        torch.cuda.synchronize()
        c = _is_canary(self.buf).cpu().numpy()
        b, n = self.band, self.n
        assert c[:b].all(), f"{what}: write before the array"
        assert c[b + n:].all(), f"{what}: write after the array"
        if written:
            assert not c[b:b + n].any(), f"{what}: {int(c[b:b + n].sum())} elements unwritten"


class BandedRows:
    """[B, L, V] rows of stride V + gap starting `head` elements into a guard buffer."""

    def __init__(self, B, L, V, dtype, head, gap=2, fill_from=None):
        self.B, self.L, self.V, self.head, self.gap = B, L, V, head, gap
        n = head + B * L * (V + gap) + BAND
        self.buf = torch.empty(n, dtype=dtype, device=DEV)
        _fill(self.buf)
        self.t = torch.as_strided(self.buf, (B, L, V), (L * (V + gap), V + gap, 1), head)
        if fill_from is not None:
            self.t.copy_(fill_from)
        cov = np.zeros(n, bool)
        for r in range(B * L):
            cov[head + r * (V + gap): head + r * (V + gap) + V] = True
        self.cov = cov

    def check(self, what):
        torch.cuda.synchronize()
        c = _is_canary(self.buf).cpu().numpy()
        out = ~self.cov
        assert c[out].all(), f"{what}: {int((~c[out]).sum())} writes outside the rows (head, gaps or tail)"
        assert not c[self.cov].any(), f"{what}: {int(c[self.cov].sum())} row elements unwritten"


def _inputs(B, L, V, dtype, head, seed):
    g = torch.Generator().manual_seed(seed)
    R = B * L
    x = BandedRows(B, L, V, dtype, head, gap=3,
                   fill_from=(torch.randn(B, L, V, generator=g) * 2.0).to(dtype).to(DEV))
    idx = torch.randint(0, V, (R,), generator=g).to(DEV)
    adv = torch.randn(B, generator=g).float()
    adv[0] = 0.0
    mask = (torch.rand(R, generator=g) > 0.3).to(torch.uint8)
    mask[0] = 0
    dloss = ((torch.rand(R, generator=g) + 0.1) * mask.float()).float()
    lp_noise = torch.randn(R, generator=g).float()
    return x, idx, adv.to(DEV), mask.to(DEV), dloss.to(DEV), lp_noise.to(DEV)


def _ok(st, fn):
    assert st == rp.GRPO_OK, f"{fn}: {rp.status_string(st)}"


def _p(t):
    return None if t is None else t.data_ptr()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("V", VS)
@pytest.mark.parametrize("head", HEADS)
def test_row_pass_entry_points_write_only_their_outputs(dtype, V, head):
    lib = rp.load_library()
    B, L = 2, 5
    R = B * L
    s = torch.cuda.current_stream().cuda_stream
    x, idx, adv, mask, dloss, noise = _inputs(B, L, V, dtype, head, V * 13 + head)
    xd = rp.rows_of(x.t)
    T, beta, el, eh = 0.9, 0.05, 0.2, 0.28
    f32 = lambda: Banded(R, torch.float32)

    # selective_log_softmax_fwd: logp, lse
    logp, lse = f32(), f32()
    _ok(lib.selective_log_softmax_fwd(ctypes.byref(xd), _p(idx), T, logp.ptr, lse.ptr, None, s), "slsm fwd")
    logp.check("slsm fwd logp")
    lse.check("slsm fwd lse")
    old = (logp.t + 0.2 * noise).contiguous()
    ref = (logp.t - 0.1 * noise).contiguous()

    # grpo_loss_fwd: every output
    o = {k: f32() for k in ("loss", "logp", "lse", "kl", "entropy")}
    o["is_clipped"] = Banded(R, torch.uint8)
    _ok(lib.grpo_loss_fwd(ctypes.byref(xd), _p(idx), _p(old), _p(ref), _p(adv), _p(mask), T, beta, el, eh,
                          o["loss"].ptr, o["logp"].ptr, o["lse"].ptr, o["kl"].ptr, o["is_clipped"].ptr,
                          o["entropy"].ptr, None, s), "grpo fwd")
    for k, b in o.items():
        b.check(f"grpo fwd {k}")

    # grpo_loss_bwd: dlogits rows out of phase with the logits rows
    dl = BandedRows(B, L, V, dtype, head + 1)
    dld = rp.rows_of(dl.t)
    _ok(lib.grpo_loss_bwd(ctypes.byref(xd), _p(idx), _p(old), _p(ref), _p(adv), _p(mask), _p(dloss),
                          _p(o["logp"].t), _p(o["lse"].t), T, beta, el, eh, ctypes.byref(dld), None, s), "grpo bwd")
    dl.check(f"grpo bwd V={V}")

    # grpo_loss_fused
    fo = {k: f32() for k in ("loss", "logp", "lse", "kl", "entropy")}
    fo["is_clipped"] = Banded(R, torch.uint8)
    fdl = BandedRows(B, L, V, dtype, head + 2)
    fdld = rp.rows_of(fdl.t)
    _ok(lib.grpo_loss_fused(ctypes.byref(xd), _p(idx), _p(old), _p(ref), _p(adv), _p(mask), _p(dloss), T, beta,
                            el, eh, fo["loss"].ptr, fo["logp"].ptr, fo["lse"].ptr, fo["kl"].ptr,
                            fo["is_clipped"].ptr, fo["entropy"].ptr, ctypes.byref(fdld), None, s), "fused")
    for k, b in fo.items():
        b.check(f"fused {k}")
    fdl.check(f"fused dlogits V={V}")

    # entropy_from_logits (with lse) and its backward
    H, H_lse = f32(), f32()
    _ok(lib.entropy_from_logits(ctypes.byref(xd), T, H.ptr, H_lse.ptr, s), "entropy")
    H.check("entropy")
    H_lse.check("entropy lse")
    up = (noise * mask.float()).contiguous()
    edl = BandedRows(B, L, V, dtype, head + 1)
    edld = rp.rows_of(edl.t)
    _ok(lib.entropy_from_logits_bwd(ctypes.byref(xd), _p(up), _p(H_lse.t), _p(H.t), T, ctypes.byref(edld), s),
        "entropy bwd")
    edl.check(f"entropy bwd V={V}")

    # selective_log_softmax_bwd
    sdl = BandedRows(B, L, V, dtype, head + 3)
    sdld = rp.rows_of(sdl.t)
    _ok(lib.selective_log_softmax_bwd(ctypes.byref(xd), _p(idx), _p(up), _p(lse.t), T, ctypes.byref(sdld), None,
                                      s), "slsm bwd")
    sdl.check(f"slsm bwd V={V}")


@pytest.mark.parametrize("V", [65541, 151936])
@pytest.mark.parametrize("head", HEADS)
@pytest.mark.parametrize("beta", [0.0, 0.05])
def test_fused_same_phase_rows_write_only_their_rows(V, head, beta):
    """grpo_loss_fused with the dlogits rows in the logits' own layout (row stride V + 3, so
    the rows start at varying 16-byte phases): the long-row launch, which holds the first
    104 KB of each row in shared memory, prefetches the rest into L2 and writes masked and
    zero rows (beta = 0, zero advantage) by bulk stores from shared memory.  Out of place,
    then in place."""
    lib = rp.load_library()
    B, L = 2, 5
    R = B * L
    s = torch.cuda.current_stream().cuda_stream
    x, idx, adv, mask, dloss, noise = _inputs(B, L, V, torch.bfloat16, head, V * 17 + head)
    xd = rp.rows_of(x.t)
    T, el, eh = 0.9, 0.2, 0.28
    logp, lse = Banded(R, torch.float32), Banded(R, torch.float32)
    _ok(lib.selective_log_softmax_fwd(ctypes.byref(xd), _p(idx), T, logp.ptr, lse.ptr, None, s), "slsm fwd")
    old = (logp.t + 0.2 * noise).contiguous()
    ref = (logp.t - 0.1 * noise).contiguous()
    for in_place in (False, True):
        fo = {k: Banded(R, torch.float32) for k in ("loss", "logp", "lse", "kl", "entropy")}
        fo["is_clipped"] = Banded(R, torch.uint8)
        fdl = x if in_place else BandedRows(B, L, V, torch.bfloat16, head, gap=3)
        fdld = rp.rows_of(fdl.t)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        _ok(lib.grpo_loss_fused(ctypes.byref(xd), _p(idx), _p(old), _p(ref), _p(adv), _p(mask), _p(dloss), T,
                                beta, el, eh, fo["loss"].ptr, fo["logp"].ptr, fo["lse"].ptr, fo["kl"].ptr,
                                fo["is_clipped"].ptr, fo["entropy"].ptr, ctypes.byref(fdld), _p(err), s), "fused")
        for k, b in fo.items():
            b.check(f"fused {k} in_place={in_place}")
        fdl.check(f"fused dlogits V={V} in_place={in_place}")
        assert int(err.item()) == 0


@pytest.mark.parametrize("V", VS)
@pytest.mark.parametrize("head", HEADS)
def test_vocab_shard_entry_points_write_only_their_outputs(V, head):
    lib = rp.load_library()
    dtype = torch.bfloat16
    B, L = 2, 5
    R = B * L
    s = torch.cuda.current_stream().cuda_stream
    x, idx, adv, mask, dloss, noise = _inputs(B, L, V, dtype, head, V * 17 + head)
    T, beta, el, eh = 1.1, 0.04, 0.2, 0.28
    cut = [0, V // 2, V] if V > 1 else [0, 1]
    world = len(cut) - 1
    stats = Banded(world * R * 4, torch.float32)
    for k in range(world):
        sh = x.t[:, :, cut[k]:cut[k + 1]]
        shd = rp.rows_of(sh)
        out = stats.t[k * R * 4:(k + 1) * R * 4]
        _ok(lib.grpo_vocab_shard_stats(ctypes.byref(shd), cut[k], _p(idx), _p(mask), T, out.data_ptr(), s), "stats")
    torch.cuda.synchronize()
    stats.check("shard stats")  # masked rows get (0, 0, 0, 0)
    starts = (ctypes.c_int64 * (world + 1))(*cut)
    logp0 = torch.randn(R, generator=torch.Generator().manual_seed(V)).float().to(DEV) - 5.0
    old = (logp0 + 0.1 * noise).contiguous()
    ref = (logp0 - 0.05 * noise).contiguous()
    o = {k: Banded(R, torch.float32) for k in ("loss", "logp", "lse", "kl", "entropy", "p_rest")}
    o["is_clipped"] = Banded(R, torch.uint8)
    _ok(lib.grpo_vocab_combine(world, stats.ptr, starts, B, L, _p(idx), _p(old), _p(ref), _p(adv), _p(mask), T,
                               beta, el, eh, o["loss"].ptr, o["logp"].ptr, o["lse"].ptr, o["kl"].ptr,
                               o["is_clipped"].ptr, o["entropy"].ptr, o["p_rest"].ptr, None, s), "combine")
    for k, b in o.items():
        b.check(f"combine {k}")
    for k in range(world):
        sh = x.t[:, :, cut[k]:cut[k + 1]]
        w = cut[k + 1] - cut[k]
        dl = BandedRows(B, L, w, dtype, head + 1)
        _ok(lib.grpo_loss_bwd_vocab_shard(ctypes.byref(rp.rows_of(sh)), cut[k], V, _p(idx), _p(old), _p(ref),
                                          _p(adv), _p(mask), _p(dloss), _p(o["logp"].t), _p(o["lse"].t),
                                          _p(o["p_rest"].t), T, beta, el, eh, ctypes.byref(rp.rows_of(dl.t)), None,
                                          s), "shard bwd")
        dl.check(f"grpo shard bwd V={V} shard {k}")
        sdl = BandedRows(B, L, w, dtype, head + 2)
        _ok(lib.selective_log_softmax_bwd_vocab_shard(ctypes.byref(rp.rows_of(sh)), cut[k], V, _p(idx), _p(dloss),
                                                      _p(o["lse"].t), _p(o["p_rest"].t), T,
                                                      ctypes.byref(rp.rows_of(sdl.t)), None, s), "slsm shard bwd")
        sdl.check(f"slsm shard bwd V={V} shard {k}")


@pytest.mark.parametrize("L", [1, 7, 1024, 1500])
def test_seq_terms_write_only_their_outputs(L):
    lib = rp.load_library()
    B = 3
    R = B * L
    s = torch.cuda.current_stream().cuda_stream
    g = torch.Generator().manual_seed(L)
    logp = (torch.randn(R, generator=g) - 4.0).float().to(DEV)
    old = (logp + 0.1 * torch.randn(R, generator=g).to(DEV)).contiguous()
    ref = (logp - 0.05 * torch.randn(R, generator=g).to(DEV)).contiguous()
    adv = torch.randn(B, generator=g).float().to(DEV)
    mask = (torch.rand(R, generator=g) > 0.2).to(torch.uint8).to(DEV)
    dloss = (mask.float() / R).contiguous()
    o = {k: Banded(R, torch.float32) for k in ("loss", "kl", "dlogp")}
    ratio, clip = Banded(B, torch.float32), Banded(B, torch.uint8)
    _ok(lib.grpo_seq_terms(B, L, _p(logp), _p(old), _p(ref), _p(adv), _p(mask), _p(dloss), 0.04, 0.2, 0.28,
                           o["loss"].ptr, o["kl"].ptr, o["dlogp"].ptr, ratio.ptr, clip.ptr, s), "seq terms")
    for k, b in o.items():
        b.check(f"seq terms {k}")
    ratio.check("seq ratio")
    clip.check("seq is_clipped")


@pytest.mark.parametrize("V", [1, 7, 9, 513, 40000])
def test_fused_linear_writes_only_its_outputs(V):
    lib = rp.load_library()
    B, L, H = 2, 9, 64
    R = B * L
    s = torch.cuda.current_stream().cuda_stream
    g = torch.Generator().manual_seed(V)
    hidden = torch.randn(R, H, generator=g).to(torch.bfloat16).to(DEV)
    weight = (torch.randn(V, H, generator=g) * 0.25).to(torch.bfloat16).to(DEV)
    idx = torch.randint(0, V, (R,), generator=g).to(DEV)
    adv = torch.randn(B, generator=g).float().to(DEV)
    mask = (torch.rand(R, generator=g) > 0.3).to(torch.uint8).to(DEV)
    dloss = (mask.float() / R).contiguous()
    chunk = 5  # several chunks and a ragged last one
    need = rp.grpo_fused_linear_workspace_size(H, V, chunk)
    ws = Banded(need, torch.uint8, band=256)  # the workspace must start 256-byte aligned
    o = {k: Banded(R, torch.float32) for k in ("loss", "logp", "lse", "kl", "entropy")}
    o["is_clipped"] = Banded(R, torch.uint8)
    gh = Banded(R * H, torch.float32)
    gw = Banded(V * H, torch.float32, zero_inside=True)
    _ok(lib.grpo_fused_linear(hidden.data_ptr(), weight.data_ptr(), B, L, H, V, _p(idx), None, None, _p(adv),
                              _p(mask), _p(dloss), 1.0, 0.0, 0.2, 0.28, chunk, ws.ptr, need, o["loss"].ptr,
                              o["logp"].ptr, o["lse"].ptr, o["kl"].ptr, o["is_clipped"].ptr, o["entropy"].ptr,
                              gh.ptr, gw.ptr, None, s), "fused linear")
    for k, b in o.items():
        b.check(f"fused linear {k}")
    gh.check("fused linear grad_hidden")
    gw.check("fused linear grad_weight")
    ws.check("fused linear workspace", written=False)
