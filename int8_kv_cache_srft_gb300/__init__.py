"""int8_kv_cache_srft_gb300 -- Python binding of libsrftkv (GB300, sm_103a).

A thin ctypes layer over the C ABI in ``include/srftkv.h``: it turns torch
tensors into device pointers and the current torch stream into a
cudaStream_t, calls the entry point of the same name and raises on a
non-zero return.  All arithmetic happens in the library's CUDA kernels;
there is no CPU or PyTorch fallback, and importing this package fails
loudly when the library has not been built (``python -m
int8_kv_cache_srft_gb300.build``).
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsrftkv.so")

SRFTKV_OK = 0
SRFTKV_ERR_INVALID = -1
SRFTKV_ERR_CUDA = -2
SRFTKV_ERR_DEVICE = -3


class SrftKvError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} returned {code}: {msg}")
        self.code = code


class _Side(ctypes.Structure):
    _fields_ = [
        ("x", ctypes.c_void_p),
        ("lambda_", ctypes.c_void_p),
        ("lambda_outer_stride", ctypes.c_int64),
        ("bits", ctypes.c_int),
        ("codes", ctypes.c_void_p),
        ("scales", ctypes.c_void_p),
        ("transform", ctypes.c_int),
        ("scale_format", ctypes.c_int),
    ]


TRANSFORMS = {"srft": 0, "srht": 1}  # SRFTKV_TRANSFORM_SRFT / _SRHT in include/srftkv.h
SCALE_FORMATS = {"fp32": 0, "fp16": 1, "e8m0": 2}  # SRFTKV_SCALE_FP32 / _FP16 / _E8M0
SCALE_DTYPES = {"fp32": torch.float32, "fp16": torch.float16, "e8m0": torch.uint8}


_lib = None


def library() -> ctypes.CDLL:
    """Load libsrftkv.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -m int8_kv_cache_srft_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    i, u64, vp, sz = ctypes.c_int, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_size_t
    sp = ctypes.POINTER(_Side)
    lib.srft_kv_quantize.argtypes = [sp, sp, i, i, i, i, i, i, i, u64, vp]
    lib.srft_kv_dequantize.argtypes = [sp, sp, i, i, i, i, i, i, i, u64, vp]
    lib.q4kv_decode_attention.argtypes = [vp, vp, sp, sp, i, i, i, i, i, i, vp, ctypes.c_float, u64, i, vp, sz, vp]
    lib.q4kv_decode_attention_static.argtypes = [vp, vp, sp, sp, i, i, i, i, i, i, vp, ctypes.c_float, u64, i, vp]
    lib.q4kv_decode_attention_workspace_size.argtypes = [i, i, i, i, i, i]
    lib.q4kv_decode_attention_workspace_size.restype = sz
    lib.srft_kv_vector_bytes.argtypes = [i, i, i, i, ctypes.POINTER(sz), ctypes.POINTER(sz)]
    lib.srft_transform.argtypes = [vp, vp, i, i, u64, i, vp]
    lib.srht_transform.argtypes = [vp, vp, i, i, u64, i, vp]
    lib.srftkv_last_error.restype = ctypes.c_char_p
    lib.srftkv_device_fault.argtypes = [ctypes.POINTER(ctypes.c_uint)]
    lib.srftkv_set_attention_poll_limit_for_testing.argtypes = [i]
    lib.srftkv_set_codec_poll_limit_for_testing.argtypes = [i]
    for name in ("srft_kv_quantize", "srft_kv_dequantize", "q4kv_decode_attention", "q4kv_decode_attention_static",
                 "srft_kv_vector_bytes", "srft_transform", "srht_transform", "srftkv_device_fault",
                 "srftkv_set_attention_poll_limit_for_testing", "srftkv_set_codec_poll_limit_for_testing"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(fn: str, rc: int) -> None:
    if rc != SRFTKV_OK:
        raise SrftKvError(fn, rc, library().srftkv_last_error().decode())


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> int | None:
    if stream is None:  # torch's current stream on the current device
        if _raw_stream is not None:
            return _raw_stream(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


@dataclass
class Side:
    """One side (K or V) of a packed cache: the code plane, the scale plane,
    an optional per-channel lambda and, for the codec calls, the fp16 rows."""

    codes: torch.Tensor            # uint8 [n_outer][H][t_cap][d*bits/8] (or fp16 [B][Hkv][t_cap][d] for bits 16)
    scales: torch.Tensor | None    # [n_outer][H][t_cap][d/group]: fp32, fp16 or uint8 (e8m0) per scale_format
    bits: int
    x: torch.Tensor | None = None  # fp16 [n_outer][n_tokens][H][d]
    lam: torch.Tensor | None = None  # fp32 [n_lam][H][d]; n_lam == 1 broadcasts
    lam_outer_stride: int | None = None
    transform: str = "srft"        # "srft" or "srht"
    scale_format: str = "fp32"     # "fp32", "fp16" or "e8m0"

    # The marshalled struct is built once and reused until a field is assigned again (a tensor changed in
    # place keeps its address; one resized or replaced must be assigned anew).
    def __setattr__(self, name, value):
        object.__setattr__(self, name, value)
        if name != "_c":
            object.__setattr__(self, "_c", None)

    def c_pointer(self):
        c = getattr(self, "_c", None)
        if c is None:
            c = ctypes.pointer(self.to_c())
            object.__setattr__(self, "_c", c)
        return c

    def to_c(self) -> _Side:
        stride = self.lam_outer_stride
        if stride is None:
            stride = 0 if self.lam is None or self.lam.shape[0] == 1 else self.lam.shape[1] * self.lam.shape[2]
        return _Side(_ptr(self.x), _ptr(self.lam), stride, self.bits, _ptr(self.codes), _ptr(self.scales),
                     TRANSFORMS[self.transform], SCALE_FORMATS[self.scale_format])


def alloc_side(n_outer: int, t_cap: int, H: int, d: int, bits: int, group: int, device="cuda",
               transform: str = "srft", scale_format: str = "fp32") -> Side:
    """Allocate empty (head-major) code and scale planes for one side."""
    if bits == 16:
        return Side(torch.empty((n_outer, H, t_cap, d), dtype=torch.float16, device=device), None, 16)
    codes = torch.empty((n_outer, H, t_cap, d * bits // 8), dtype=torch.uint8, device=device)
    scales = torch.empty((n_outer, H, t_cap, d // group), dtype=SCALE_DTYPES[scale_format], device=device)
    return Side(codes, scales, bits, transform=transform, scale_format=scale_format)


def _sidep(s: Side | None):
    return None if s is None else s.c_pointer()


def srft_kv_quantize(k: Side | None, v: Side | None, n_outer: int, n_tokens: int, H: int, d: int, group: int,
                     t_cap: int, t_offset: int, sign_seed: int, stream=None) -> None:
    rc = library().srft_kv_quantize(_sidep(k), _sidep(v), n_outer, n_tokens, H, d, group, t_cap, t_offset,
                                    sign_seed, _stream(stream))
    _check("srft_kv_quantize", rc)


def srft_kv_dequantize(k: Side | None, v: Side | None, n_outer: int, n_tokens: int, H: int, d: int, group: int,
                       t_cap: int, t_offset: int, sign_seed: int, stream=None) -> None:
    rc = library().srft_kv_dequantize(_sidep(k), _sidep(v), n_outer, n_tokens, H, d, group, t_cap, t_offset,
                                      sign_seed, _stream(stream))
    _check("srft_kv_dequantize", rc)


def q4kv_decode_attention_workspace_size(B: int, Hq: int, Hkv: int, d: int, t_cap: int, n_splits: int = 0) -> int:
    return int(library().q4kv_decode_attention_workspace_size(B, Hq, Hkv, d, t_cap, n_splits))


def q4kv_decode_attention(q: torch.Tensor, out: torch.Tensor, k: Side, v: Side, B: int, Hq: int, Hkv: int, d: int,
                          group: int, t_cap: int, seq_lens: torch.Tensor | None, sm_scale: float, sign_seed: int,
                          n_splits: int, workspace: torch.Tensor, stream=None) -> None:
    rc = library().q4kv_decode_attention(_ptr(q), _ptr(out), _sidep(k), _sidep(v), B, Hq, Hkv, d, group, t_cap,
                                         _ptr(seq_lens), sm_scale, sign_seed, n_splits, _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), _stream(stream))
    _check("q4kv_decode_attention", rc)


STATIC_SCRATCH_BYTES = 16 << 20  # SRFTKV_STATIC_SCRATCH_BYTES in include/srftkv.h


def q4kv_decode_attention_static(q: torch.Tensor, out: torch.Tensor, k: Side, v: Side, B: int, Hq: int, Hkv: int,
                                 d: int, group: int, t_cap: int, seq_lens: torch.Tensor | None, sm_scale: float,
                                 sign_seed: int, n_splits: int, stream=None) -> None:
    """Decode attention without a caller workspace, for callers that cannot allocate device memory: the
    library's own fixed-size device array is the scratch (see include/srftkv.h for its size and the rules on
    overlapping calls)."""
    rc = library().q4kv_decode_attention_static(_ptr(q), _ptr(out), _sidep(k), _sidep(v), B, Hq, Hkv, d, group,
                                                t_cap, _ptr(seq_lens), sm_scale, sign_seed, n_splits,
                                                _stream(stream))
    _check("q4kv_decode_attention_static", rc)


def srft_kv_vector_bytes(d: int, bits: int, group: int, scale_format: str = "fp32") -> tuple[int, int]:
    """(code bytes, scale bytes) of one packed vector."""
    cb, sb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    fmt = SCALE_FORMATS[scale_format] if isinstance(scale_format, str) else int(scale_format)
    _check("srft_kv_vector_bytes", library().srft_kv_vector_bytes(d, bits, group, fmt, ctypes.byref(cb),
                                                                  ctypes.byref(sb)))
    return cb.value, sb.value


def srft_transform(x: torch.Tensor, y: torch.Tensor, n: int, d: int, sign_seed: int, inverse: bool,
                   stream=None) -> None:
    rc = library().srft_transform(_ptr(x), _ptr(y), n, d, sign_seed, int(bool(inverse)), _stream(stream))
    _check("srft_transform", rc)


def srht_transform(x: torch.Tensor, y: torch.Tensor, n: int, d: int, sign_seed: int, inverse: bool,
                   stream=None) -> None:
    rc = library().srht_transform(_ptr(x), _ptr(y), n, d, sign_seed, int(bool(inverse)), _stream(stream))
    _check("srht_transform", rc)


def srftkv_device_fault() -> int:
    f = ctypes.c_uint(0)
    _check("srftkv_device_fault", library().srftkv_device_fault(ctypes.byref(f)))
    return f.value


def srftkv_set_attention_poll_limit_for_testing(polls: int) -> None:
    """Test hook: polls of the attention kernel's chunk wait before a warp gives up (negative = the default,
    0 = give up at the first chunk)."""
    _check("srftkv_set_attention_poll_limit_for_testing",
           library().srftkv_set_attention_poll_limit_for_testing(int(polls)))


def srftkv_set_codec_poll_limit_for_testing(polls: int) -> None:
    """Test hook: polls of the register-path quantize kernels' tile wait before a warp gives up (negative = the
    default, 0 = give up at the first tile)."""
    _check("srftkv_set_codec_poll_limit_for_testing",
           library().srftkv_set_codec_poll_limit_for_testing(int(polls)))


def srftkv_last_error() -> str:
    return library().srftkv_last_error().decode()
