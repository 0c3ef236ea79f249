"""Python binding of the C ABI in ``include/cpattn.h`` (ctypes; argument marshalling only).

Every function here validates tensor shapes/dtypes just enough to build the C call, allocates
output tensors when the caller passes none, and calls the library on the current torch CUDA
stream.  All computation happens in the CUDA kernels of ``libcpattn.so``; there is no fallback.
If the library is missing or cannot be loaded, the first call raises ``CpAttnLibraryError``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

__all__ = ["CpAttnError", "CpAttnLibraryError", "lib", "attn_fwd", "attn_fwd_chunked",
           "attn_lse_merge", "attn_fwd_ulysses", "attn_fwd_ring", "attn_fwd_fp8", "cp_absmax",
           "cp_quantize_e4m3", "cp_layout_seq2head",
           "cp_layout_head2seq", "attn_device_status",
           "attn_watchdog_selftest", "attn_set_max_ctas", "attn_probe_mma", "attn_probe_alu",
           "attn_set_kernel_variant", "attn_status_string", "attn_version",
           "LIB_PATH", "ATTN_OK", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_UNSUPPORTED",
           "ATTN_ERR_MISALIGNED", "ATTN_ERR_CUDA", "ATTN_ERR_TIMEOUT"]

# CPATTN_LIBRARY may point at another build of the same library (e.g. a debug build).
LIB_PATH = os.environ.get("CPATTN_LIBRARY") or os.path.join(
    os.path.dirname(os.path.abspath(__file__)), "libcpattn.so")

ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED = 0, 1, 2
ATTN_ERR_MISALIGNED, ATTN_ERR_CUDA, ATTN_ERR_TIMEOUT = 3, 4, 5
_DT = {torch.bfloat16: 0, torch.float16: 1}


class CpAttnLibraryError(RuntimeError):
    pass


class CpAttnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {attn_status_string(status)} ({status})")


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded ``libcpattn.so`` with argument types declared."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise CpAttnLibraryError(
            f"{LIB_PATH} is not built; run `python -m context_math_non_b300.build`")
    try:
        L = ctypes.CDLL(LIB_PATH)
    except OSError as e:
        raise CpAttnLibraryError(f"cannot load {LIB_PATH}: {e}") from e
    vp, i, f, fp = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_void_p
    L.attn_fwd.argtypes = [vp, vp, vp, vp, fp, i, i, i, i, i, i, f, vp]
    L.attn_fwd_chunked.argtypes = [vp, vp, vp, i, vp, fp, i, i, i, i, i, i, f, vp]
    L.attn_lse_merge.argtypes = [vp, fp, i, i, i, i, i, i, vp, fp, vp]
    L.attn_fwd_ulysses.argtypes = [vp, vp, vp, vp, fp, i, i, i, i, i, i, f, vp]
    L.attn_fwd_ring.argtypes = [vp, vp, vp, i, vp, fp, i, i, i, i, i, i, f, vp]
    L.attn_fwd_fp8.argtypes = [vp, vp, vp, i, f, f, f, vp, fp, i, i, i, i, i, f, vp]
    L.cp_absmax.argtypes = [vp, ctypes.c_longlong, i, fp, vp]
    L.cp_quantize_e4m3.argtypes = [vp, i, vp, i, i, i, f, i, vp]
    L.cp_layout_seq2head.argtypes = [vp, vp, i, i, i, i, i, i, vp]
    L.cp_layout_head2seq.argtypes = [vp, vp, i, i, i, i, i, i, vp]
    L.attn_status_string.argtypes = [i]
    L.attn_status_string.restype = ctypes.c_char_p
    L.attn_device_status.argtypes = [vp]
    L.attn_watchdog_selftest.argtypes = [ctypes.c_uint64, vp]
    L.attn_set_max_ctas.argtypes = [i]
    L.attn_set_kernel_variant.argtypes = [i]
    L.attn_probe_mma.argtypes = [i, i, i, vp]
    L.attn_probe_alu.argtypes = [i, i, vp]
    L.attn_version.argtypes = []
    for name in ("attn_fwd", "attn_fwd_chunked", "attn_lse_merge", "attn_fwd_ulysses",
                 "attn_fwd_ring", "attn_fwd_fp8", "cp_absmax", "cp_quantize_e4m3",
                 "cp_layout_seq2head", "cp_layout_head2seq",
                 "attn_device_status", "attn_watchdog_selftest", "attn_set_max_ctas",
                 "attn_version", "attn_probe_mma", "attn_probe_alu", "attn_set_kernel_variant"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def attn_status_string(status: int) -> str:
    return lib().attn_status_string(int(status)).decode()


def attn_version() -> int:
    return lib().attn_version()


def attn_set_max_ctas(n: int) -> int:
    return lib().attn_set_max_ctas(int(n))


def attn_set_kernel_variant(v: int) -> int:
    """0: single-CTA kernel (default); 1: D = 128 attention on SM pairs.  Returns the previous."""
    return lib().attn_set_kernel_variant(int(v))


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _check(fn: str, status: int):
    if status != ATTN_OK:
        raise CpAttnError(fn, status)


def _dev(t: torch.Tensor, name: str) -> int:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _ptr_or_null(t: Optional[torch.Tensor], name: str):
    return None if t is None else _dev(t, name)


def _dt(t: torch.Tensor, name: str) -> int:
    """Library dtype code of a 16-bit float tensor."""
    if t.dtype not in _DT:
        raise ValueError(f"{name} must be bfloat16 or float16, not {t.dtype}")
    return _DT[t.dtype]


_BYTE_TYPES = (torch.uint8,) + ((torch.float8_e4m3fn,) if hasattr(torch, "float8_e4m3fn") else ())


def _e4m3(t: torch.Tensor, name: str) -> int:
    """Pointer of a tensor of e4m3 bytes (uint8 or float8_e4m3fn)."""
    if t.dtype not in _BYTE_TYPES:
        raise ValueError(f"{name} must hold e4m3 bytes (uint8 or float8_e4m3fn), not {t.dtype}")
    return _dev(t, name)


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: Optional[torch.Tensor] = None,
             lse: Optional[torch.Tensor] = None, scale: float = 0.0, want_lse: bool = True,
             stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """O, LSE of non-causal attention; q [B,H,Sq,D], k/v [B,H,Skv,D] (bf16 or fp16)."""
    B, H, Sq, D = q.shape
    Skv = k.shape[2]
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    _check("attn_fwd", lib().attn_fwd(
        _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(o, "o"), _ptr_or_null(lse, "lse"),
        B, H, Sq, Skv, D, _dt(q, "q"), float(scale), _stream(stream)))
    return o, lse


def attn_fwd_chunked(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, P: int,
                     o_parts: Optional[torch.Tensor] = None,
                     lse_parts: Optional[torch.Tensor] = None, scale: float = 0.0,
                     stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Per-KV-chunk partials: O_parts [P,B,H,Sq,D], LSE_parts [P,B,H,Sq] fp32."""
    B, H, Sq, D = q.shape
    Skv = k.shape[2]
    if o_parts is None:
        o_parts = torch.empty((P, B, H, Sq, D), dtype=q.dtype, device=q.device)
    if lse_parts is None:
        lse_parts = torch.empty((P, B, H, Sq), dtype=torch.float32, device=q.device)
    _check("attn_fwd_chunked", lib().attn_fwd_chunked(
        _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), int(P), _dev(o_parts, "o_parts"),
        _dev(lse_parts, "lse_parts"), B, H, Sq, Skv, D, _dt(q, "q"), float(scale),
        _stream(stream)))
    return o_parts, lse_parts


def attn_lse_merge(o_parts: torch.Tensor, lse_parts: torch.Tensor,
                   o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                   want_lse: bool = True, stream=None):
    """Merge partials [P,B,H,Sq,D] / [P,B,H,Sq] into O [B,H,Sq,D] and LSE [B,H,Sq]."""
    P, B, H, Sq, D = o_parts.shape
    if o is None:
        o = torch.empty((B, H, Sq, D), dtype=o_parts.dtype, device=o_parts.device)
    if lse is None and want_lse:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=o_parts.device)
    _check("attn_lse_merge", lib().attn_lse_merge(
        _dev(o_parts, "o_parts"), _dev(lse_parts, "lse_parts"), P, B, H, Sq, D,
        _dt(o_parts, "o_parts"), _dev(o, "o"), _ptr_or_null(lse, "lse"), _stream(stream)))
    return o, lse


def attn_fwd_ring(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, P: int,
                  o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                  scale: float = 0.0, want_lse: bool = True, stream=None):
    """Ring attention over P KV chunks with the merge fused in: O [B,H,Sq,D], LSE [B,H,Sq]."""
    B, H, Sq, D = q.shape
    Skv = k.shape[2]
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    _check("attn_fwd_ring", lib().attn_fwd_ring(
        _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), P, _dev(o, "o"), _ptr_or_null(lse, "lse"),
        B, H, Sq, Skv, D, _dt(q, "q"), float(scale), _stream(stream)))
    return o, lse


def attn_fwd_fp8(q8: torch.Tensor, k8: torch.Tensor, vt8: torch.Tensor, P: int, q_scale: float,
                 k_scale: float, v_scale: float, o: Optional[torch.Tensor] = None,
                 lse: Optional[torch.Tensor] = None, scale: float = 0.0, want_lse: bool = True,
                 stream=None):
    """e4m3 attention: q8 [B,H,Sq,D], k8 [B,H,Skv,D], vt8 [B,H,D,Skv] (one byte per element);
    O bf16 [B,H,Sq,D], LSE [B,H,Sq]."""
    B, H, Sq, D = q8.shape
    Skv = k8.shape[2]
    if o is None:
        o = torch.empty((B, H, Sq, D), dtype=torch.bfloat16, device=q8.device)
    if lse is None and want_lse:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q8.device)
    _check("attn_fwd_fp8", lib().attn_fwd_fp8(
        _e4m3(q8, "q"), _e4m3(k8, "k"), _e4m3(vt8, "vt"), P, float(q_scale), float(k_scale),
        float(v_scale), _dev(o, "o"), _ptr_or_null(lse, "lse"), B, H, Sq, Skv, D, float(scale),
        _stream(stream)))
    return o, lse


def cp_absmax(x: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """max |x| of a bf16/fp16 tensor, as a one-element fp32 device tensor."""
    if out is None:
        out = torch.empty((1,), dtype=torch.float32, device=x.device)
    _check("cp_absmax", lib().cp_absmax(_dev(x, "x"), x.numel(), _dt(x, "x"), _dev(out, "amax"),
                                        _stream(stream)))
    return out


def cp_quantize_e4m3(x: torch.Tensor, scale: float, transpose: bool = False,
                     out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """e4m3 bytes of x / scale: x [..., S, D] -> [..., S, D], or [..., D, S] when transpose."""
    *lead, S, D = x.shape
    BH = 1
    for d in lead:
        BH *= d
    if out is None:
        shape = (*lead, D, S) if transpose else (*lead, S, D)
        out = torch.empty(shape, dtype=torch.uint8, device=x.device)
    _check("cp_quantize_e4m3", lib().cp_quantize_e4m3(
        _dev(x, "x"), _dt(x, "x"), _dev(out, "y"), BH, S, D, float(scale), int(transpose),
        _stream(stream)))
    return out


def attn_fwd_ulysses(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                     o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                     scale: float = 0.0, want_lse: bool = True, stream=None):
    """Ulysses attention on sequence-sharded q/k/v [P][B][S/P][H][D]; O in the same layout,
    LSE [P][B][H/P][S] fp32."""
    P, B, Sl, H, D = q.shape
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((P, B, H // P, Sl * P), dtype=torch.float32, device=q.device)
    _check("attn_fwd_ulysses", lib().attn_fwd_ulysses(
        _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(o, "o"), _ptr_or_null(lse, "lse"),
        P, B, Sl * P, H, D, _dt(q, "q"), float(scale), _stream(stream)))
    return o, lse


def cp_layout_seq2head(x: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None):
    """[P][B][S/P][H][D] -> [P][B][H/P][S][D] (first Ulysses all-to-all)."""
    P, B, Sl, H, D = x.shape
    if out is None:
        out = torch.empty((P, B, H // P, Sl * P, D), dtype=x.dtype, device=x.device)
    _check("cp_layout_seq2head", lib().cp_layout_seq2head(
        _dev(x, "in"), _dev(out, "out"), P, B, Sl * P, H, D, x.element_size(), _stream(stream)))
    return out


def cp_layout_head2seq(y: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None):
    """[P][B][H/P][S][D] -> [P][B][S/P][H][D] (second Ulysses all-to-all)."""
    P, B, Hl, S, D = y.shape
    if out is None:
        out = torch.empty((P, B, S // P, Hl * P, D), dtype=y.dtype, device=y.device)
    _check("cp_layout_head2seq", lib().cp_layout_head2seq(
        _dev(y, "in"), _dev(out, "out"), P, B, S, Hl * P, D, y.element_size(), _stream(stream)))
    return out


def attn_probe_mma(n: int, mode: int, iters: int, stream=None):
    """Launch the tensor-core ceiling probe (time it with CUDA events around the call)."""
    _check("attn_probe_mma", lib().attn_probe_mma(int(n), int(mode), int(iters),
                                                   _stream(stream)))


def attn_probe_alu(mode: int, iters: int, stream=None):
    _check("attn_probe_alu", lib().attn_probe_alu(int(mode), int(iters), _stream(stream)))


def attn_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the kernels' status word."""
    return lib().attn_device_status(_stream(stream))


def attn_watchdog_selftest(limit_ns: int, stream=None):
    _check("attn_watchdog_selftest", lib().attn_watchdog_selftest(int(limit_ns), _stream(stream)))
