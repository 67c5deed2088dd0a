"""Thin ctypes binding over libfa_gb300.so (include/fa.h).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels. PyTorch supplies device memory and the current
stream. Importing this module raises ImportError when the library has not
been built (there is no fallback path).
"""

from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa_gb300.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -m io_aware_exact_fa_gb300.build` "
        "(or __graft_entry__.build()); there is no non-CUDA fallback")

_lib = ctypes.CDLL(LIB_PATH)

_vp = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64
_u64 = ctypes.c_uint64
_f = ctypes.c_float
_sz = ctypes.c_size_t

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT, FA_ERR_WORKSPACE = range(6)

EXPORTS = {
    "fa_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp]),
    "fa_fwd_masked": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp, _i64, _i64, _i64, _vp]),
    "fa_fwd_fp8": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _f, _f, _f, _i, _vp]),
    "fa_fwd_host_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i]),
    "fa_fwd_host": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _i, _vp, _sz, _vp]),
    "fa_decode_workspace_size": (_sz, [_i, _i, _i, _i]),
    "fa_decode_splitkv": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _sz, _vp]),
    "fa_decode_splitkv_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp]),
    "fa_decode_grouped_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
    "fa_decode_grouped": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _sz, _vp]),
    "fa_materialized_workspace_size": (_sz, [_i, _i, _i, _i]),
    "fa_fwd_materialized": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp, _sz, _vp]),
    "fa_bwd_workspace_size": (_sz, [_i, _i, _i, _i]),
    "fa_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp, _sz, _vp]),
    "fa_get_device_status": (_i, [_vp]),
    "fa_set_wait_limit_ns": (None, [_u64]),
    "fa_get_wait_limit_ns": (_u64, []),
    "fa_selftest_wait_timeout": (_i, [_u64, _vp]),
    "fa_selftest_exp2": (_i, [_vp, _vp, _i, _vp]),
    "fa_status_string": (ctypes.c_char_p, [_i]),
    "fa_last_error_detail": (ctypes.c_char_p, []),
    "fa_launch_count": (_u64, []),
    "fa_debug_enabled": (_i, []),
    "fa_debug_record": (_i, [_vp, _vp]),
    "fa_debug_selftest": (_i, [_vp]),
}
for _name, (_res, _args) in EXPORTS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


def debug_library() -> ctypes.CDLL:
    """The device-checking build (libfa_gb300_debug.so, FA_DEBUG=1; see
    include/fa.h), with the same entry points as the release library. Build it
    with ``build.build(debug=True)``."""
    path = os.path.join(_HERE, "libfa_gb300_debug.so")
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -m io_aware_exact_fa_gb300.build --debug`")
    dl = ctypes.CDLL(path)
    for name, (res, args) in EXPORTS.items():
        fn = getattr(dl, name)
        fn.restype = res
        fn.argtypes = args
    return dl


class FAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = _lib.fa_last_error_detail().decode()
        super().__init__(f"{where}: {_lib.fa_status_string(status).decode()} {detail}".strip())


def _check(status: int, where: str) -> None:
    if status != FA_OK:
        raise FAError(status, where)


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype=torch.bfloat16) -> None:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: Optional[float] = None,
        causal: bool = False, keep_bits: Optional[torch.Tensor] = None,
        mask_strides: Tuple[int, int, int] = (0, 0, 0), out: Optional[torch.Tensor] = None,
        lse: Optional[torch.Tensor] = None, with_lse: bool = True,
        stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Exact attention forward pass: q [B,H,Nq,d], k/v [B,H,Nk,d] bf16 -> (o bf16, lse fp32).

    ``keep_bits`` (int32 words, bit j%32 of word j//32 = key j, 1 = attend)
    with ``mask_strides`` = (b, h, q) strides in words; q stride 0 broadcasts.
    """
    _need(q, "q"); _need(k, "k"); _need(v, "v")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if k.shape != (B, H, Nk, d) or v.shape != (B, H, Nk, d):
        raise ValueError("k and v must be [B, H, Nk, d] matching q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out")
    if with_lse and lse is None:
        lse = torch.empty(B, H, Nq, dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32)
    st = _stream_ptr(stream)
    lp = lse.data_ptr() if lse is not None else None
    if keep_bits is None:
        rc = _lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lp,
                         B, H, Nq, Nk, d, float(scale), int(bool(causal)), st)
        _check(rc, "fa_fwd")
    else:
        _need(keep_bits, "keep_bits", torch.int32)
        sb, sh, sq = mask_strides
        rc = _lib.fa_fwd_masked(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lp,
                                B, H, Nq, Nk, d, float(scale), int(bool(causal)),
                                keep_bits.data_ptr(), int(sb), int(sh), int(sq), st)
        _check(rc, "fa_fwd_masked")
    return out, lse


def fwd_fp8(q8: torch.Tensor, k8: torch.Tensor, v8: torch.Tensor, descale_q: float, descale_k: float,
            descale_v: float, scale: Optional[float] = None, causal: bool = False,
            out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None, with_lse: bool = True,
            stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Forward pass on e4m3 inputs (fa_fwd_fp8): q8 [B,H,Nq,d], k8/v8 [B,H,Nk,d]
    as uint8 codes (or torch.float8_e4m3fn), each with one descale factor
    (real value = code value * descale) -> (o bf16, lse fp32)."""
    q8, k8, v8 = (t.view(torch.uint8) if isinstance(t, torch.Tensor) and t.dtype == torch.float8_e4m3fn else t
                  for t in (q8, k8, v8))
    _need(q8, "q8", torch.uint8); _need(k8, "k8", torch.uint8); _need(v8, "v8", torch.uint8)
    B, H, Nq, d = q8.shape
    Nk = k8.shape[2]
    if k8.shape != (B, H, Nk, d) or v8.shape != (B, H, Nk, d):
        raise ValueError("k8 and v8 must be [B, H, Nk, d] matching q8")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(B, H, Nq, d, dtype=torch.bfloat16, device=q8.device)
    _need(out, "out")
    if with_lse and lse is None:
        lse = torch.empty(B, H, Nq, dtype=torch.float32, device=q8.device)
    if lse is not None:
        _need(lse, "lse", torch.float32)
    rc = _lib.fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), out.data_ptr(),
                         lse.data_ptr() if lse is not None else None, B, H, Nq, Nk, d, float(scale),
                         float(descale_q), float(descale_k), float(descale_v), int(bool(causal)),
                         _stream_ptr(stream))
    _check(rc, "fa_fwd_fp8")
    return out, lse


def fwd_host_workspace_size(B: int, H: int, Nq: int, Nk: int, d: int, chunk_heads: int = 0) -> int:
    return int(_lib.fa_fwd_host_workspace_size(B, H, Nq, Nk, d, chunk_heads))


def _need_host(t: torch.Tensor, name: str, dtype=torch.bfloat16) -> None:
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: Optional[float] = None,
             causal: bool = False, chunk_heads: int = 0, workspace: Optional[torch.Tensor] = None,
             out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None, with_lse: bool = True,
             stream: Optional[torch.cuda.Stream] = None,
             sync: bool = True) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """fa_fwd_host: the forward pass on HOST tensors (q [B,H,Nq,d], k/v [B,H,Nk,d]
    bf16; pin them for overlap). The library copies chunks of heads to the
    current CUDA device, runs the fused kernel there and copies o and lse
    back. With ``sync`` the call waits for ``stream`` before returning;
    otherwise the host outputs are complete once the stream is synchronised."""
    _need_host(q, "q"); _need_host(k, "k"); _need_host(v, "v")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if k.shape != (B, H, Nk, d) or v.shape != (B, H, Nk, d):
        raise ValueError("k and v must be [B, H, Nk, d] matching q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    pin = q.is_pinned()
    if out is None:
        out = torch.empty(tuple(q.shape), dtype=q.dtype, pin_memory=pin)
    _need_host(out, "out")
    if with_lse and lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, pin_memory=pin)
    if lse is not None:
        _need_host(lse, "lse", torch.float32)
    if workspace is None:
        workspace = torch.empty(max(1, fwd_host_workspace_size(B, H, Nq, Nk, d, chunk_heads)), dtype=torch.uint8,
                                device="cuda")
    _need(workspace, "workspace", torch.uint8)
    st = _stream_ptr(stream)
    rc = _lib.fa_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                          lse.data_ptr() if lse is not None else None, B, H, Nq, Nk, d, float(scale),
                          int(bool(causal)), int(chunk_heads), workspace.data_ptr(),
                          workspace.numel(), st)
    _check(rc, "fa_fwd_host")
    if sync:
        (stream if stream is not None else torch.cuda.current_stream()).synchronize()
    return out, lse


def decode_workspace_size(B: int, H: int, d: int, num_splits: int) -> int:
    return int(_lib.fa_decode_workspace_size(B, H, d, num_splits))


def decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, scale: Optional[float] = None,
           num_splits: int = 16, workspace: Optional[torch.Tensor] = None,
           out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None, with_lse: bool = True,
           stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Split-KV decode: q [B,H,1,d], caches [B,H,Nk,d] bf16 -> (o [B,H,1,d] bf16, lse [B,H] fp32)."""
    _need(q, "q"); _need(k_cache, "k_cache"); _need(v_cache, "v_cache")
    B, H, one, d = q.shape
    if one != 1:
        raise ValueError("decode takes one query token per (b, h): q must be [B, H, 1, d]")
    Nk = k_cache.shape[2]
    if k_cache.shape != (B, H, Nk, d) or v_cache.shape != (B, H, Nk, d):
        raise ValueError("k_cache and v_cache must be [B, H, Nk, d]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = decode_workspace_size(B, H, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out")
    if with_lse and lse is None:
        lse = torch.empty(B, H, dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32)
    rc = _lib.fa_decode_splitkv(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(),
                                lse.data_ptr() if lse is not None else None, B, H, Nk, d, float(scale),
                                int(num_splits), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                _stream_ptr(stream))
    _check(rc, "fa_decode_splitkv")
    return out, lse


def decode_grouped_workspace_size(B: int, H: int, Nq: int, d: int, num_splits: int) -> int:
    return int(_lib.fa_decode_grouped_workspace_size(B, H, Nq, d, num_splits))


def decode_grouped(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                   seqlens_k: Optional[torch.Tensor] = None, scale: Optional[float] = None, num_splits: int = 8,
                   workspace: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                   lse: Optional[torch.Tensor] = None, with_lse: bool = True,
                   stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Decode with grouped K/V heads, Nq new tokens and per-sequence lengths (fa.h fa_decode_grouped):
    q [B,H,Nq,d], caches [B,Hkv,Nk,d] bf16, seqlens_k int32 [B] or None -> (o [B,H,Nq,d], lse [B,H,Nq])."""
    _need(q, "q"); _need(k_cache, "k_cache"); _need(v_cache, "v_cache")
    B, H, Nq, d = q.shape
    Hkv, Nk = k_cache.shape[1], k_cache.shape[2]
    if k_cache.shape != (B, Hkv, Nk, d) or v_cache.shape != (B, Hkv, Nk, d):
        raise ValueError("k_cache and v_cache must be [B, Hkv, Nk, d]")
    if seqlens_k is not None:
        _need(seqlens_k, "seqlens_k", torch.int32)
        if seqlens_k.shape != (B,):
            raise ValueError("seqlens_k must be int32 [B]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = decode_grouped_workspace_size(B, H, Nq, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out")
    if with_lse and lse is None:
        lse = torch.empty(B, H, Nq, dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32)
    rc = _lib.fa_decode_grouped(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                seqlens_k.data_ptr() if seqlens_k is not None else None, out.data_ptr(),
                                lse.data_ptr() if lse is not None else None, B, H, Hkv, Nq, Nk, d, float(scale),
                                int(num_splits), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                _stream_ptr(stream))
    _check(rc, "fa_decode_grouped")
    return out, lse


NOALLOC_SCRATCH_BYTES = 20 << 20


def decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, scale: Optional[float] = None,
                   num_splits: int = 16, out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                   with_lse: bool = True, stream: Optional[torch.cuda.Stream] = None):
    """Split-KV decode using the library's static scratch (no workspace); see fa.h."""
    _need(q, "q"); _need(k_cache, "k_cache"); _need(v_cache, "v_cache")
    B, H, one, d = q.shape
    if one != 1:
        raise ValueError("decode takes one query token per (b, h): q must be [B, H, 1, d]")
    Nk = k_cache.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if with_lse and lse is None:
        lse = torch.empty(B, H, dtype=torch.float32, device=q.device)
    rc = _lib.fa_decode_splitkv_noalloc(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(),
                                        lse.data_ptr() if lse is not None else None, B, H, Nk, d, float(scale),
                                        int(num_splits), _stream_ptr(stream))
    _check(rc, "fa_decode_splitkv_noalloc")
    return out, lse


def materialized_workspace_size(B: int, H: int, Nq: int, Nk: int) -> int:
    return int(_lib.fa_materialized_workspace_size(B, H, Nq, Nk))


def fwd_materialized(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: Optional[float] = None,
                     causal: bool = False, workspace: Optional[torch.Tensor] = None,
                     out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                     stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """The materialising baseline (fa.h fa_fwd_materialized): S and P through HBM in bf16."""
    _need(q, "q"); _need(k, "k"); _need(v, "v")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if k.shape != (B, H, Nk, d) or v.shape != (B, H, Nk, d):
        raise ValueError("k and v must be [B, H, Nk, d]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = materialized_workspace_size(B, H, Nq, Nk)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, H, Nq, dtype=torch.float32, device=q.device)
    _need(out, "out"); _need(lse, "lse", torch.float32)
    rc = _lib.fa_fwd_materialized(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, Nq,
                                  Nk, d, float(scale), int(bool(causal)), workspace.data_ptr(),
                                  workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _check(rc, "fa_fwd_materialized")
    return out, lse


def bwd_workspace_size(B: int, H: int, Nq: int, d: int) -> int:
    return int(_lib.fa_bwd_workspace_size(B, H, Nq, d))


def bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, lse: torch.Tensor,
        dout: torch.Tensor, scale: Optional[float] = None, causal: bool = False,
        workspace: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None,
        grads: Optional[Tuple[torch.Tensor, torch.Tensor, torch.Tensor]] = None):
    """Backward pass of ``fwd`` (no key mask): returns (dq, dk, dv), bf16, shaped like q, k, v
    (written into ``grads`` when given)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        _need(t, n)
    _need(lse, "lse", torch.float32)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if k.shape != (B, H, Nk, d) or v.shape != (B, H, Nk, d) or o.shape != q.shape or dout.shape != q.shape:
        raise ValueError("shapes: q, o, dout [B,H,Nq,d]; k, v [B,H,Nk,d]")
    if lse.shape != (B, H, Nq):
        raise ValueError("lse must be [B, H, Nq]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = bwd_workspace_size(B, H, Nq, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if grads is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    else:
        dq, dk, dv = grads
        for t, ref, n in ((dq, q, "dq"), (dk, k, "dk"), (dv, v, "dv")):
            _need(t, n)
            if t.shape != ref.shape:
                raise ValueError(f"{n} must be shaped like its input")
    rc = _lib.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                     dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Nq, Nk, d, float(scale), int(bool(causal)),
                     workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _check(rc, "fa_bwd")
    return dq, dk, dv


def device_status(stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronise and return (then clear) the library's device status (FA_OK or FA_ERR_TIMEOUT)."""
    return int(_lib.fa_get_device_status(_stream_ptr(stream)))


def selftest_wait_timeout(limit_ns: int, stream: Optional[torch.cuda.Stream] = None) -> int:
    return int(_lib.fa_selftest_wait_timeout(int(limit_ns), _stream_ptr(stream)))


def selftest_exp2(x: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """2^x through the device FMA-pipe exponential used inside the prefill softmax."""
    _need(x, "x", torch.float32)
    y = torch.empty_like(x)
    _check(_lib.fa_selftest_exp2(x.data_ptr(), y.data_ptr(), x.numel(), _stream_ptr(stream)), "fa_selftest_exp2")
    return y


def set_wait_limit_ns(ns: int) -> None:
    _lib.fa_set_wait_limit_ns(int(ns))


def get_wait_limit_ns() -> int:
    return int(_lib.fa_get_wait_limit_ns())


def launch_count() -> int:
    return int(_lib.fa_launch_count())


def status_string(s: int) -> str:
    return _lib.fa_status_string(s).decode()


# raw handle for callers that pass their own pointers (host-buffer end-to-end timing, tests)
lib = _lib
