"""Thin Python binding over the C ABI in ``include/grpo_rowpass.h``.

Argument marshalling only: each function checks tensor devices/dtypes, allocates the
outputs with torch (device memory is torch's job here), and calls the C entry point of
the same name on the current CUDA stream.  Every step of the row pass runs in the CUDA
kernels of ``libgrpo_rowpass.so``; there is no CPU fallback.  A missing library raises
``RuntimeError`` on first use.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from .build import LIB_PATH

GRPO_OK, GRPO_ERR_INVALID_ARG, GRPO_ERR_UNSUPPORTED, GRPO_ERR_CUDA = 0, 1, 2, 3
GRPO_FP32, GRPO_BF16 = 0, 1
GRPO_DEVERR_IDX_OUT_OF_RANGE = 1

EXPORTED = ("grpo_loss_fwd", "grpo_loss_bwd", "grpo_loss_fused", "entropy_from_logits",
            "entropy_from_logits_bwd", "selective_log_softmax_fwd", "selective_log_softmax_bwd",
            "grpo_seq_terms", "grpo_vocab_shard_stats", "grpo_vocab_combine", "grpo_loss_bwd_vocab_shard",
            "selective_log_softmax_bwd_vocab_shard", "grpo_fused_linear_workspace_size", "grpo_fused_linear",
            "grpo_fused_linear_noalloc", "grpo_status_string")
GRPO_VOCAB_MAX_WORLD = 64


class GrpoRows(ctypes.Structure):
    """Mirror of ``grpo_rows``."""
    _fields_ = [("ptr", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("B", ctypes.c_int64), ("L", ctypes.c_int64), ("V", ctypes.c_int64),
                ("stride_b", ctypes.c_int64), ("stride_l", ctypes.c_int64)]


class GrpoError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)}")


_lib = None
_P = ctypes.c_void_p
_F = ctypes.c_float


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load ``libgrpo_rowpass.so`` (once) and declare the C signatures."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m rl_fine_tuning_pass_gb300.build` "
                           "(or __graft_entry__.build()); the row pass has no fallback")
    lib = ctypes.CDLL(path)
    rows_p = ctypes.POINTER(GrpoRows)
    sig = {
        "grpo_loss_fwd": [rows_p, _P, _P, _P, _P, _P, _F, _F, _F, _F, _P, _P, _P, _P, _P, _P, _P, _P],
        "grpo_loss_bwd": [rows_p, _P, _P, _P, _P, _P, _P, _P, _P, _F, _F, _F, _F, rows_p, _P, _P],
        "grpo_loss_fused": [rows_p, _P, _P, _P, _P, _P, _P, _F, _F, _F, _F, _P, _P, _P, _P, _P, _P, rows_p, _P, _P],
        "entropy_from_logits": [rows_p, _F, _P, _P, _P],
        "entropy_from_logits_bwd": [rows_p, _P, _P, _P, _F, rows_p, _P],
        "grpo_seq_terms": [ctypes.c_int64, ctypes.c_int64, _P, _P, _P, _P, _P, _P, _F, _F, _F, _P, _P, _P, _P, _P, _P],
        "selective_log_softmax_fwd": [rows_p, _P, _F, _P, _P, _P, _P],
        "selective_log_softmax_bwd": [rows_p, _P, _P, _P, _F, rows_p, _P, _P],
        "grpo_vocab_shard_stats": [rows_p, ctypes.c_int64, _P, _P, _F, _P, _P],
        "grpo_vocab_combine": [ctypes.c_int32, _P, _P, ctypes.c_int64, ctypes.c_int64, _P, _P, _P, _P, _P,
                               _F, _F, _F, _F, _P, _P, _P, _P, _P, _P, _P, _P, _P],
        "grpo_loss_bwd_vocab_shard": [rows_p, ctypes.c_int64, ctypes.c_int64, _P, _P, _P, _P, _P, _P, _P, _P,
                                      _P, _F, _F, _F, _F, rows_p, _P, _P],
        "selective_log_softmax_bwd_vocab_shard": [rows_p, ctypes.c_int64, ctypes.c_int64, _P, _P, _P, _P, _F,
                                                  rows_p, _P, _P],
        "grpo_fused_linear_workspace_size": [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                             ctypes.POINTER(ctypes.c_uint64)],
        "grpo_fused_linear": [_P, _P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _P, _P, _P, _P,
                              _P, _P, _F, _F, _F, _F, ctypes.c_int64, _P, ctypes.c_uint64, _P, _P, _P, _P, _P, _P,
                              _P, _P, _P, _P],
        "grpo_fused_linear_noalloc": [_P, _P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _P, _P,
                                      _P, _P, _P, _P, _F, _F, _F, _F, ctypes.c_int64, _P, _P, _P, _P, _P, _P, _P, _P,
                                      _P, _P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.grpo_status_string.argtypes = [ctypes.c_int]
    lib.grpo_status_string.restype = ctypes.c_char_p
    if path == LIB_PATH:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().grpo_status_string(int(status)).decode()


def rows_of(t: torch.Tensor) -> GrpoRows:
    """Describe a [B, L, V] (or [R, V], read as B=1, L=R) tensor with vocab stride 1."""
    if t.dim() == 2:
        B, L, V = 1, t.shape[0], t.shape[1]
        sb, sl = t.shape[0] * t.stride(0), t.stride(0)
    elif t.dim() == 3:
        B, L, V = t.shape
        sb, sl = t.stride(0), t.stride(1)
    else:
        raise ValueError("logits must be [B, L, V] or [R, V]")
    if V > 0 and t.stride(-1) != 1:
        raise ValueError("the vocabulary dimension must have stride 1")
    if t.dtype == torch.bfloat16:
        dt = GRPO_BF16
    elif t.dtype == torch.float32:
        dt = GRPO_FP32
    else:
        raise TypeError(f"logits dtype {t.dtype} not supported (bf16 or fp32)")
    return GrpoRows(t.data_ptr(), dt, 0, B, L, V, sb, sl)


def _ptr(t: Optional[torch.Tensor], dtype, n: Optional[int], name: str):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if n is not None and t.numel() != n:
        raise ValueError(f"{name} must have {n} elements, got {t.numel()}")
    return t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _check(fn: str, st: int):
    if st != GRPO_OK:
        raise GrpoError(fn, st)


def _shape(logits: torch.Tensor):
    if not logits.is_cuda:
        raise ValueError("logits must be a CUDA tensor")
    if logits.dim() == 3:
        return logits.shape[0], logits.shape[1]
    return 1, logits.shape[0]


def grpo_loss_fwd(logits, idx, adv, *, T, beta, eps_low, eps_high, old_logp=None, ref_logp=None,
                  mask=None, with_kl=True, with_is_clipped=True, with_entropy=False, dev_err=None):
    """GRPO forward; returns a dict with loss, logp, lse (+ kl, is_clipped, entropy)."""
    B, L = _shape(logits)
    R = B * L
    dev = logits.device
    f32 = dict(dtype=torch.float32, device=dev)
    out = {"loss": torch.empty(R, **f32), "logp": torch.empty(R, **f32), "lse": torch.empty(R, **f32)}
    out["kl"] = torch.empty(R, **f32) if with_kl else None
    out["is_clipped"] = torch.empty(R, dtype=torch.uint8, device=dev) if with_is_clipped else None
    out["entropy"] = torch.empty(R, **f32) if with_entropy else None
    x = rows_of(logits)
    st = load_library().grpo_loss_fwd(
        ctypes.byref(x), _ptr(idx, torch.int64, R, "idx"), _ptr(old_logp, torch.float32, R, "old_logp"),
        _ptr(ref_logp, torch.float32, R, "ref_logp"), _ptr(adv, torch.float32, B, "adv"),
        _ptr(mask, torch.uint8, R, "mask"), float(T), float(beta), float(eps_low), float(eps_high),
        out["loss"].data_ptr(), out["logp"].data_ptr(), out["lse"].data_ptr(),
        _ptr(out["kl"], torch.float32, R, "kl"), _ptr(out["is_clipped"], torch.uint8, R, "is_clipped"),
        _ptr(out["entropy"], torch.float32, R, "entropy"), _ptr(dev_err, torch.int32, 1, "dev_err"),
        _stream(dev))
    _check("grpo_loss_fwd", st)
    return {k: v for k, v in out.items() if v is not None}


def grpo_loss_bwd(logits, idx, adv, dloss, logp, lse, *, T, beta, eps_low, eps_high, old_logp=None,
                  ref_logp=None, mask=None, dlogits=None, dev_err=None):
    """GRPO backward; returns dlogits (allocated [B, L, V] like logits unless given;
    pass ``dlogits=logits`` for an in-place backward)."""
    B, L = _shape(logits)
    R = B * L
    if dlogits is None:
        dlogits = torch.empty(logits.shape, dtype=logits.dtype, device=logits.device)
    x, dx = rows_of(logits), rows_of(dlogits)
    st = load_library().grpo_loss_bwd(
        ctypes.byref(x), _ptr(idx, torch.int64, R, "idx"), _ptr(old_logp, torch.float32, R, "old_logp"),
        _ptr(ref_logp, torch.float32, R, "ref_logp"), _ptr(adv, torch.float32, B, "adv"),
        _ptr(mask, torch.uint8, R, "mask"), _ptr(dloss, torch.float32, R, "dloss"),
        _ptr(logp, torch.float32, R, "logp"), _ptr(lse, torch.float32, R, "lse"), float(T), float(beta),
        float(eps_low), float(eps_high), ctypes.byref(dx), _ptr(dev_err, torch.int32, 1, "dev_err"),
        _stream(logits.device))
    _check("grpo_loss_bwd", st)
    return dlogits


def grpo_loss_fused(logits, idx, adv, dloss, *, T, beta, eps_low, eps_high, old_logp=None, ref_logp=None,
                    mask=None, with_kl=True, with_is_clipped=True, with_entropy=False, dlogits=None, dev_err=None):
    """GRPO forward and backward in one pass (dloss known in advance); returns the forward's
    dict plus "dlogits"."""
    B, L = _shape(logits)
    R = B * L
    dev = logits.device
    f32 = dict(dtype=torch.float32, device=dev)
    out = {"loss": torch.empty(R, **f32), "logp": torch.empty(R, **f32), "lse": torch.empty(R, **f32)}
    out["kl"] = torch.empty(R, **f32) if with_kl else None
    out["is_clipped"] = torch.empty(R, dtype=torch.uint8, device=dev) if with_is_clipped else None
    out["entropy"] = torch.empty(R, **f32) if with_entropy else None
    if dlogits is None:
        dlogits = torch.empty(logits.shape, dtype=logits.dtype, device=dev)
    x, dx = rows_of(logits), rows_of(dlogits)
    st = load_library().grpo_loss_fused(
        ctypes.byref(x), _ptr(idx, torch.int64, R, "idx"), _ptr(old_logp, torch.float32, R, "old_logp"),
        _ptr(ref_logp, torch.float32, R, "ref_logp"), _ptr(adv, torch.float32, B, "adv"),
        _ptr(mask, torch.uint8, R, "mask"), _ptr(dloss, torch.float32, R, "dloss"), float(T), float(beta),
        float(eps_low), float(eps_high), out["loss"].data_ptr(), out["logp"].data_ptr(), out["lse"].data_ptr(),
        _ptr(out["kl"], torch.float32, R, "kl"), _ptr(out["is_clipped"], torch.uint8, R, "is_clipped"),
        _ptr(out["entropy"], torch.float32, R, "entropy"), ctypes.byref(dx),
        _ptr(dev_err, torch.int32, 1, "dev_err"), _stream(dev))
    _check("grpo_loss_fused", st)
    res = {k: v for k, v in out.items() if v is not None}
    res["dlogits"] = dlogits
    return res


def entropy_from_logits(logits, *, T=1.0, return_lse=False):
    """Per-row entropy [B*L] fp32 (and lse [B*L] when return_lse)."""
    B, L = _shape(logits)
    out = torch.empty(B * L, dtype=torch.float32, device=logits.device)
    lse = torch.empty(B * L, dtype=torch.float32, device=logits.device) if return_lse else None
    x = rows_of(logits)
    st = load_library().entropy_from_logits(ctypes.byref(x), float(T), out.data_ptr(),
                                            None if lse is None else lse.data_ptr(), _stream(logits.device))
    _check("entropy_from_logits", st)
    return (out, lse) if return_lse else out


def entropy_from_logits_bwd(logits, dentropy, lse, entropy, *, T=1.0, dlogits=None):
    """dlogits of sum_r dentropy_r * H_r (allocated like logits unless given)."""
    B, L = _shape(logits)
    R = B * L
    if dlogits is None:
        dlogits = torch.empty(logits.shape, dtype=logits.dtype, device=logits.device)
    x, dx = rows_of(logits), rows_of(dlogits)
    st = load_library().entropy_from_logits_bwd(
        ctypes.byref(x), _ptr(dentropy, torch.float32, R, "dentropy"), _ptr(lse, torch.float32, R, "lse"),
        _ptr(entropy, torch.float32, R, "entropy"), float(T), ctypes.byref(dx), _stream(logits.device))
    _check("entropy_from_logits_bwd", st)
    return dlogits


def selective_log_softmax_fwd(logits, idx, *, T=1.0, dev_err=None):
    """Returns (logp, lse), each [B*L] fp32."""
    B, L = _shape(logits)
    R = B * L
    logp = torch.empty(R, dtype=torch.float32, device=logits.device)
    lse = torch.empty(R, dtype=torch.float32, device=logits.device)
    x = rows_of(logits)
    st = load_library().selective_log_softmax_fwd(
        ctypes.byref(x), _ptr(idx, torch.int64, R, "idx"), float(T), logp.data_ptr(), lse.data_ptr(),
        _ptr(dev_err, torch.int32, 1, "dev_err"), _stream(logits.device))
    _check("selective_log_softmax_fwd", st)
    return logp, lse


def selective_log_softmax_bwd(logits, idx, dlogp, lse, *, T=1.0, dlogits=None, dev_err=None):
    """Returns dlogits of sum_r dlogp_r * logp_r (allocated like logits unless given)."""
    B, L = _shape(logits)
    R = B * L
    if dlogits is None:
        dlogits = torch.empty(logits.shape, dtype=logits.dtype, device=logits.device)
    x, dx = rows_of(logits), rows_of(dlogits)
    st = load_library().selective_log_softmax_bwd(
        ctypes.byref(x), _ptr(idx, torch.int64, R, "idx"), _ptr(dlogp, torch.float32, R, "dlogp"),
        _ptr(lse, torch.float32, R, "lse"), float(T), ctypes.byref(dx), _ptr(dev_err, torch.int32, 1, "dev_err"),
        _stream(logits.device))
    _check("selective_log_softmax_bwd", st)
    return dlogits


def grpo_seq_terms(logp, adv, dloss, *, B, L, beta, eps_low, eps_high, old_logp=None, ref_logp=None, mask=None):
    """Sequence-level GRPO terms; returns dict(loss, kl, dlogp [B*L], seq_ratio [B],
    seq_is_clipped [B]).  Feed dlogp to selective_log_softmax_bwd for the dlogits."""
    R = B * L
    dev = logp.device
    f32 = dict(dtype=torch.float32, device=dev)
    out = {"loss": torch.empty(R, **f32), "kl": torch.empty(R, **f32), "dlogp": torch.empty(R, **f32),
           "seq_ratio": torch.empty(B, **f32), "seq_is_clipped": torch.empty(B, dtype=torch.uint8, device=dev)}
    st = load_library().grpo_seq_terms(
        B, L, _ptr(logp, torch.float32, R, "logp"), _ptr(old_logp, torch.float32, R, "old_logp"),
        _ptr(ref_logp, torch.float32, R, "ref_logp"), _ptr(adv, torch.float32, B, "adv"),
        _ptr(mask, torch.uint8, R, "mask"), _ptr(dloss, torch.float32, R, "dloss"), float(beta), float(eps_low),
        float(eps_high), out["loss"].data_ptr(), out["kl"].data_ptr(), out["dlogp"].data_ptr(),
        out["seq_ratio"].data_ptr(), out["seq_is_clipped"].data_ptr(), _stream(dev))
    _check("grpo_seq_terms", st)
    return out


# ---------------------------------------------------------------------------
# vocabulary-parallel form (each rank holds a column shard of every row)
# ---------------------------------------------------------------------------

def grpo_vocab_shard_stats(logits_shard, vocab_start, *, T=1.0, idx=None, mask=None):
    """Per-row statistic (a, s, u, x_sel) of one vocabulary shard: [B*L, 4] fp32."""
    B, L = _shape(logits_shard)
    R = B * L
    stats = torch.empty(R, 4, dtype=torch.float32, device=logits_shard.device)
    x = rows_of(logits_shard)
    st = load_library().grpo_vocab_shard_stats(
        ctypes.byref(x), int(vocab_start), _ptr(idx, torch.int64, R, "idx"), _ptr(mask, torch.uint8, R, "mask"),
        float(T), stats.data_ptr(), _stream(logits_shard.device))
    _check("grpo_vocab_shard_stats", st)
    return stats


def grpo_vocab_combine(stats_all, vocab_starts, B, L, *, T=1.0, idx=None, adv=None, grpo=False, beta=0.0,
                       eps_low=0.2, eps_high=0.2, old_logp=None, ref_logp=None, mask=None, with_entropy=True,
                       with_p_rest=True, dev_err=None):
    """Merge gathered shard statistics [world, B*L, 4] (rank order) into the full rows'
    outputs: dict with lse (+ entropy), and with idx given logp and p_rest, and with
    grpo=True the GRPO terms (loss, kl, is_clipped)."""
    world = int(stats_all.shape[0])
    R = B * L
    dev = stats_all.device
    if stats_all.dtype != torch.float32 or tuple(stats_all.shape) != (world, R, 4) or not stats_all.is_contiguous():
        raise ValueError("stats_all must be a contiguous [world, B*L, 4] float32 tensor")
    if not stats_all.is_cuda:
        raise ValueError("stats_all must be a CUDA tensor")
    starts = (ctypes.c_int64 * (world + 1))(*[int(v) for v in vocab_starts])
    if len(vocab_starts) != world + 1:
        raise ValueError("vocab_starts needs world + 1 entries")
    f32 = dict(dtype=torch.float32, device=dev)
    out = {"lse": torch.empty(R, **f32), "entropy": torch.empty(R, **f32) if with_entropy else None,
           "logp": None, "p_rest": None, "loss": None, "kl": None, "is_clipped": None}
    if idx is not None:
        out["logp"] = torch.empty(R, **f32)
        out["p_rest"] = torch.empty(R, **f32) if with_p_rest else None
    if grpo:
        out["loss"], out["kl"] = torch.empty(R, **f32), torch.empty(R, **f32)
        out["is_clipped"] = torch.empty(R, dtype=torch.uint8, device=dev)
    p = lambda k, dt=torch.float32: _ptr(out[k], dt, R, k)
    st = load_library().grpo_vocab_combine(
        world, stats_all.data_ptr(), starts, B, L, _ptr(idx, torch.int64, R, "idx"),
        _ptr(old_logp, torch.float32, R, "old_logp"), _ptr(ref_logp, torch.float32, R, "ref_logp"),
        _ptr(adv, torch.float32, B, "adv"), _ptr(mask, torch.uint8, R, "mask"), float(T), float(beta),
        float(eps_low), float(eps_high), p("loss"), p("logp"), p("lse"), p("kl"), p("is_clipped", torch.uint8),
        p("entropy"), p("p_rest"), _ptr(dev_err, torch.int32, 1, "dev_err"), _stream(dev))
    _check("grpo_vocab_combine", st)
    return {k: v for k, v in out.items() if v is not None}


def grpo_loss_bwd_vocab_shard(logits_shard, vocab_start, vocab_total, idx, adv, dloss, logp, lse, p_rest, *, T,
                              beta, eps_low, eps_high, old_logp=None, ref_logp=None, mask=None, dlogits=None,
                              dev_err=None):
    """This shard's columns of the GRPO dlogits (allocated like logits_shard unless given)."""
    B, L = _shape(logits_shard)
    R = B * L
    if dlogits is None:
        dlogits = torch.empty(logits_shard.shape, dtype=logits_shard.dtype, device=logits_shard.device)
    x, dx = rows_of(logits_shard), rows_of(dlogits)
    st = load_library().grpo_loss_bwd_vocab_shard(
        ctypes.byref(x), int(vocab_start), int(vocab_total), _ptr(idx, torch.int64, R, "idx"),
        _ptr(old_logp, torch.float32, R, "old_logp"), _ptr(ref_logp, torch.float32, R, "ref_logp"),
        _ptr(adv, torch.float32, B, "adv"), _ptr(mask, torch.uint8, R, "mask"), _ptr(dloss, torch.float32, R, "dloss"),
        _ptr(logp, torch.float32, R, "logp"), _ptr(lse, torch.float32, R, "lse"),
        _ptr(p_rest, torch.float32, R, "p_rest"), float(T), float(beta), float(eps_low), float(eps_high),
        ctypes.byref(dx), _ptr(dev_err, torch.int32, 1, "dev_err"), _stream(logits_shard.device))
    _check("grpo_loss_bwd_vocab_shard", st)
    return dlogits


def selective_log_softmax_bwd_vocab_shard(logits_shard, vocab_start, vocab_total, idx, dlogp, lse, p_rest, *,
                                          T=1.0, dlogits=None, dev_err=None):
    """This shard's columns of the selective-log-softmax dlogits."""
    B, L = _shape(logits_shard)
    R = B * L
    if dlogits is None:
        dlogits = torch.empty(logits_shard.shape, dtype=logits_shard.dtype, device=logits_shard.device)
    x, dx = rows_of(logits_shard), rows_of(dlogits)
    st = load_library().selective_log_softmax_bwd_vocab_shard(
        ctypes.byref(x), int(vocab_start), int(vocab_total), _ptr(idx, torch.int64, R, "idx"),
        _ptr(dlogp, torch.float32, R, "dlogp"), _ptr(lse, torch.float32, R, "lse"),
        _ptr(p_rest, torch.float32, R, "p_rest"), float(T), ctypes.byref(dx),
        _ptr(dev_err, torch.int32, 1, "dev_err"), _stream(logits_shard.device))
    _check("selective_log_softmax_bwd_vocab_shard", st)
    return dlogits


# ---------------------------------------------------------------------------
# the GRPO loss on top of the LM head (hidden states and head weight)
# ---------------------------------------------------------------------------

def grpo_fused_linear_workspace_size(H, V, chunk_rows):
    out = ctypes.c_uint64(0)
    _check("grpo_fused_linear_workspace_size",
           load_library().grpo_fused_linear_workspace_size(int(H), int(V), int(chunk_rows), ctypes.byref(out)))
    return int(out.value)


def grpo_fused_linear(hidden, weight, idx, adv, dloss, *, B, L, T, beta, eps_low, eps_high, old_logp=None,
                      ref_logp=None, mask=None, chunk_rows=2048, with_grad_hidden=True, grad_weight=None,
                      with_grad_weight=True, with_entropy=True, workspace=None, dev_err=None):
    """GRPO loss on top of the LM head, in chunks of rows: dict with the forward outputs
    (loss, logp, lse, kl, is_clipped, entropy), grad_hidden [B*L, H] fp32 and grad_weight
    [V, H] fp32 (accumulated into the given tensor, else into zeros).  The chunks hold only
    unmasked rows.  chunk_rows trades workspace (one chunk's 16-bit exponentials / dlogits,
    statistics and gathered hidden rows, ~2.1 V + 2 H bytes a row, plus 128 MiB) for speed:
    with V = 151936, H = 1024 and 16384 rows (11180 unmasked), chunks of 2048 rows took
    8.9 ms on GB300."""
    R, H = hidden.shape
    V = weight.shape[0]
    if R != B * L:
        raise ValueError("hidden must be [B*L, H]")
    for name, t in (("hidden", hidden), ("weight", weight)):
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.shape[-1] != H:
            raise ValueError(f"{name} must be a contiguous CUDA bf16 tensor with H columns")
    dev = hidden.device
    f32 = dict(dtype=torch.float32, device=dev)
    out = {"loss": torch.empty(R, **f32), "logp": torch.empty(R, **f32), "lse": torch.empty(R, **f32),
           "kl": torch.empty(R, **f32), "is_clipped": torch.empty(R, dtype=torch.uint8, device=dev),
           "entropy": torch.empty(R, **f32) if with_entropy else None,
           "grad_hidden": torch.empty(R, H, **f32) if with_grad_hidden else None}
    if with_grad_weight and grad_weight is None:
        grad_weight = torch.zeros(V, H, **f32)
    out["grad_weight"] = grad_weight if with_grad_weight else None
    chunk = max(1, min(int(chunk_rows), R)) if R else 1
    need = grpo_fused_linear_workspace_size(H, V, chunk)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    st = load_library().grpo_fused_linear(
        hidden.data_ptr(), weight.data_ptr(), B, L, H, V, _ptr(idx, torch.int64, R, "idx"),
        _ptr(old_logp, torch.float32, R, "old_logp"), _ptr(ref_logp, torch.float32, R, "ref_logp"),
        _ptr(adv, torch.float32, B, "adv"), _ptr(mask, torch.uint8, R, "mask"), _ptr(dloss, torch.float32, R, "dloss"),
        float(T), float(beta), float(eps_low), float(eps_high), chunk, workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), out["loss"].data_ptr(), out["logp"].data_ptr(),
        out["lse"].data_ptr(), out["kl"].data_ptr(), out["is_clipped"].data_ptr(),
        _ptr(out["entropy"], torch.float32, R, "entropy"), _ptr(out["grad_hidden"], torch.float32, R * H, "grad_hidden"),
        _ptr(out["grad_weight"], torch.float32, V * H, "grad_weight"), _ptr(dev_err, torch.int32, 1, "dev_err"),
        _stream(dev))
    _check("grpo_fused_linear", st)
    return {k: v for k, v in out.items() if v is not None}
