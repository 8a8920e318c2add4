"""CPU-side checks of the C ABI: the library loads, exports every function the
header declares, computes the host-only sizes, and rejects bad arguments with
SRFTKV_ERR_INVALID before touching the GPU (so these run without one)."""

import ctypes
import os
import re

import pytest

import int8_kv_cache_srft_gb300 as K

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "srftkv.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(K.LIB_PATH):
        from int8_kv_cache_srft_gb300 import build

        build.build()
    return K.library()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s+\**([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = header_functions()
    for n in ("srft_kv_quantize", "srft_kv_dequantize", "q4kv_decode_attention",
              "q4kv_decode_attention_workspace_size", "q4kv_decode_attention_static", "srft_kv_vector_bytes",
              "srft_transform", "srht_transform", "srftkv_last_error", "srftkv_device_fault",
              "srftkv_set_attention_poll_limit_for_testing", "srftkv_set_codec_poll_limit_for_testing"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in header_functions():
        assert hasattr(lib, n), f"libsrftkv.so does not export {n}"


@pytest.mark.parametrize("d,bits,group,code,scale", [(128, 4, 16, 64, 32), (128, 8, 16, 128, 32), (256, 4, 32, 128, 32),
                                                     (16, 4, 16, 8, 4), (64, 8, 64, 64, 4), (80, 4, 16, 40, 20),
                                                     (80, 8, 16, 80, 20), (96, 4, 32, 48, 12)])
def test_vector_bytes(lib, d, bits, group, code, scale):
    assert K.srft_kv_vector_bytes(d, bits, group) == (code, scale)


@pytest.mark.parametrize("d,bits,group", [(48, 4, 16), (128, 3, 16), (128, 4, 8), (128, 4, 24), (64, 4, 128),
                                          (80, 4, 32)])
def test_vector_bytes_rejects(lib, d, bits, group):
    with pytest.raises(K.SrftKvError) as e:
        K.srft_kv_vector_bytes(d, bits, group)
    assert e.value.code == K.SRFTKV_ERR_INVALID


@pytest.mark.parametrize("d,bits,group,fmt,code,scale", [
    (128, 4, 16, "fp16", 64, 16), (128, 4, 16, "e8m0", 64, 8), (128, 8, 32, "fp16", 128, 8),
    (256, 4, 32, "e8m0", 128, 8), (96, 4, 16, "fp16", 48, 12), (192, 4, 16, "e8m0", 96, 12)])
def test_vector_bytes_scale_formats(lib, d, bits, group, fmt, code, scale):
    """The scale plane's bytes follow the scale format (4, 2 or 1 bytes a group): d=128, int4, group 16 gives
    64 + 16 = 80 bytes with fp16 scales and 64 + 8 = 72 with e8m0 (3.2x and 3.56x against 256 bytes of fp16)."""
    assert K.srft_kv_vector_bytes(d, bits, group, fmt) == (code, scale)


def test_vector_bytes_rejects_unknown_scale_format(lib):
    cb, sb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert lib.srft_kv_vector_bytes(128, 4, 16, 3, ctypes.byref(cb), ctypes.byref(sb)) == K.SRFTKV_ERR_INVALID
    assert b"scale_format" in lib.srftkv_last_error()


def _side(bits=4, x=16, codes=256, scales=256, lam=None, stride=0):
    return K._Side(x, lam, stride, bits, codes, scales)


def _q(lib, k, v, n_outer=1, n_tokens=4, H=2, d=128, group=16, t_cap=8, t_offset=0):
    kp = None if k is None else ctypes.pointer(k)
    vp = None if v is None else ctypes.pointer(v)
    return lib.srft_kv_quantize(kp, vp, n_outer, n_tokens, H, d, group, t_cap, t_offset, 1, None)


@pytest.mark.parametrize("case", [
    dict(d=100), dict(d=512), dict(d=72), dict(group=8), dict(group=48), dict(group=256), dict(d=80, group=32),
    dict(t_offset=5), dict(t_offset=-1), dict(n_tokens=-1), dict(H=0),
])
def test_quantize_rejects_bad_sizes(lib, case):
    assert _q(lib, _side(), _side(), **case) == K.SRFTKV_ERR_INVALID
    assert lib.srftkv_last_error()


def test_quantize_rejects_bad_sides(lib):
    assert _q(lib, None, None) == K.SRFTKV_ERR_INVALID
    assert _q(lib, _side(bits=3), None) == K.SRFTKV_ERR_INVALID
    assert _q(lib, _side(codes=0), None) == K.SRFTKV_ERR_INVALID
    assert _q(lib, _side(codes=8), None) == K.SRFTKV_ERR_INVALID       # misaligned code plane
    assert _q(lib, _side(scales=4), None) == K.SRFTKV_ERR_INVALID      # misaligned scale plane
    assert _q(lib, _side(x=0), None) == K.SRFTKV_ERR_INVALID
    assert _q(lib, _side(lam=4), None) == K.SRFTKV_ERR_INVALID         # misaligned lambda
    assert _q(lib, _side(lam=16, stride=6), None) == K.SRFTKV_ERR_INVALID
    # an empty call with valid arguments is a no-op and needs no GPU
    assert _q(lib, _side(), _side(), n_tokens=0) == K.SRFTKV_OK
    assert _q(lib, _side(), _side(), n_outer=0) == K.SRFTKV_OK


def test_dequantize_rejects_bad_sizes(lib):
    kp = ctypes.pointer(_side())
    assert lib.srft_kv_dequantize(kp, None, 1, 9, 2, 128, 16, 8, 0, 1, None) == K.SRFTKV_ERR_INVALID


def _attn(lib, k, v, B=2, Hq=8, Hkv=2, d=128, group=16, t_cap=64, ws=16, ws_bytes=1 << 20, q=16, out=16):
    return lib.q4kv_decode_attention(q, out, ctypes.pointer(k), ctypes.pointer(v), B, Hq, Hkv, d, group, t_cap,
                                     None, 0.0, 1, 0, ws, ws_bytes, None)


@pytest.mark.parametrize("case", [
    dict(d=32), dict(d=72), dict(Hq=6, Hkv=4), dict(B=70000, Hq=1, Hkv=1), dict(group=64), dict(t_cap=0), dict(q=0),
    dict(out=8), dict(d=80, group=32), dict(d=80, t_cap=66),
])
def test_attention_rejects_bad_arguments(lib, case):
    assert _attn(lib, _side(), _side(), **case) == K.SRFTKV_ERR_INVALID


def test_attention_rejects_mixed_raw_and_packed(lib):
    assert _attn(lib, _side(bits=16), _side(bits=4)) == K.SRFTKV_ERR_INVALID
    assert _attn(lib, _side(bits=4), _side(bits=2)) == K.SRFTKV_ERR_INVALID


def test_workspace_size_is_monotone_in_splits(lib):
    f = lib.q4kv_decode_attention_workspace_size
    s1, s8 = f(16, 32, 8, 128, 131072, 1), f(16, 32, 8, 128, 131072, 8)
    assert 0 < s1 < s8
    assert s8 >= 16 * 32 * (128 + 8 * 130) * 4
    assert f(16, 30, 8, 128, 1024, 1) == 0  # Hq not a multiple of Hkv


def test_sides_reject_unknown_transform_and_scale_format(lib):
    bad_t = _side()
    bad_t.transform = 2
    assert _q(lib, bad_t, None) == K.SRFTKV_ERR_INVALID
    bad_f = _side()
    bad_f.scale_format = 7
    assert _q(lib, None, bad_f) == K.SRFTKV_ERR_INVALID
    assert b"scale_format" in lib.srftkv_last_error()


def test_srht_transform_rejects_bad_arguments(lib):
    assert lib.srht_transform(16, 16, 4, 48, 1, 0, None) == K.SRFTKV_ERR_INVALID
    assert lib.srht_transform(None, 16, 4, 64, 1, 0, None) == K.SRFTKV_ERR_INVALID
    assert lib.srht_transform(16, 16, 0, 64, 1, 0, None) == K.SRFTKV_OK


def test_attention_format_rules(lib):
    e8 = _side()
    e8.scale_format = 2  # e8m0: 8 bytes of scales a token at d=128, group 16 -> t_cap must be even
    assert _attn(lib, e8, _side(), t_cap=63) == K.SRFTKV_ERR_INVALID
    assert b"multiple of 16" in lib.srftkv_last_error()
    bad = _side()
    bad.scale_format = 3
    assert _attn(lib, _side(), bad) == K.SRFTKV_ERR_INVALID
    bad_t = _side()
    bad_t.transform = 5
    assert _attn(lib, bad_t, _side()) == K.SRFTKV_ERR_INVALID
    assert _attn(lib, _side(scales=20), _side()) == K.SRFTKV_ERR_INVALID  # scales not 16-byte aligned


def test_attention_empty_batch_is_a_no_op(lib):
    assert _attn(lib, _side(), _side(), B=0) == K.SRFTKV_OK


@pytest.mark.parametrize("d,bits,group,code,scale", [(96, 4, 16, 48, 24), (96, 8, 32, 96, 12)])
def test_vector_bytes_d96(lib, d, bits, group, code, scale):
    assert K.srft_kv_vector_bytes(d, bits, group) == (code, scale)


def test_d96_rules(lib):
    """d = 96: groups must divide d (16 or 32), the Hadamard variant needs a power of two, and the planes are
    copied by TMA so codes and scales must be 16-byte aligned."""
    assert _q(lib, _side(), None, d=96, group=64) == K.SRFTKV_ERR_INVALID
    srht = _side()
    srht.transform = 1
    assert _q(lib, srht, None, d=96) == K.SRFTKV_ERR_INVALID
    assert b"power-of-two" in lib.srftkv_last_error()
    assert _q(lib, _side(scales=264), None, d=96) == K.SRFTKV_ERR_INVALID   # 8-byte aligned only
    assert lib.srht_transform(16, 16, 4, 96, 1, 0, None) == K.SRFTKV_ERR_INVALID
    assert lib.srft_transform(16, 16, 0, 96, 1, 0, None) == K.SRFTKV_OK
    assert _q(lib, _side(), None, d=96, n_tokens=0) == K.SRFTKV_OK


@pytest.mark.parametrize("d,bits,group,code,scale", [(192, 4, 16, 96, 48), (192, 8, 64, 192, 12)])
def test_vector_bytes_d192(lib, d, bits, group, code, scale):
    assert K.srft_kv_vector_bytes(d, bits, group) == (code, scale)


def test_d192_rules(lib):
    """d = 192: groups must divide d (16, 32 or 64; not 128), the Hadamard variant needs a power of two, codes
    and scales must be 16-byte aligned, and attention takes groups of 16 or 32 (at most d/4)."""
    assert _q(lib, _side(), None, d=192, group=128) == K.SRFTKV_ERR_INVALID
    srht = _side()
    srht.transform = 1
    assert _q(lib, srht, None, d=192) == K.SRFTKV_ERR_INVALID
    assert b"power-of-two" in lib.srftkv_last_error()
    assert _q(lib, _side(scales=264), None, d=192) == K.SRFTKV_ERR_INVALID   # 8-byte aligned only
    assert lib.srht_transform(16, 16, 4, 192, 1, 0, None) == K.SRFTKV_ERR_INVALID
    assert lib.srft_transform(16, 16, 0, 192, 1, 0, None) == K.SRFTKV_OK
    assert _q(lib, _side(), None, d=192, n_tokens=0) == K.SRFTKV_OK
    assert _attn(lib, _side(), _side(), d=192, group=64) == K.SRFTKV_ERR_INVALID


def test_side_marshalling_is_cached_until_a_field_changes():
    """The binding builds a side's C struct once; assigning any field rebuilds it with the new pointers."""
    import torch

    codes, scales = torch.zeros(64, dtype=torch.uint8), torch.zeros(8)
    s = K.Side(codes, scales, 4)
    p = s.c_pointer()
    assert s.c_pointer() is p
    assert p.contents.codes == codes.data_ptr() and p.contents.x is None
    x = torch.zeros(128, dtype=torch.float16)
    s.x = x
    q = s.c_pointer()
    assert q is not p and q.contents.x == x.data_ptr()
    lam = torch.ones((1, 2, 64))
    s.lam = lam
    r = s.c_pointer()
    assert r.contents.lambda_ == lam.data_ptr() and r.contents.lambda_outer_stride == 0
    s.scale_format = "e8m0"
    assert s.c_pointer().contents.scale_format == 2


def _attn_static(lib, k, v, B=2, Hq=8, Hkv=2, d=128, group=16, t_cap=64, n_splits=0, q=16, out=16):
    return lib.q4kv_decode_attention_static(q, out, ctypes.pointer(k), ctypes.pointer(v), B, Hq, Hkv, d, group,
                                            t_cap, None, 0.0, 1, n_splits, None)


def test_static_attention_checks_arguments_before_the_array_size(lib):
    """A bad argument is reported as itself even when the sizes would also overflow the static array, and the
    checks run before any device work (so this needs no GPU)."""
    assert _attn_static(lib, _side(), _side(), d=100, t_cap=1 << 24, n_splits=4096) == K.SRFTKV_ERR_INVALID
    assert b"d must be" in lib.srftkv_last_error()
    assert _attn_static(lib, _side(bits=3), _side(), t_cap=1 << 24, n_splits=4096) == K.SRFTKV_ERR_INVALID
    assert b"bits" in lib.srftkv_last_error()
    assert _attn_static(lib, _side(), _side(), B=0) == K.SRFTKV_OK


def test_static_scratch_size_matches_the_header():
    """The binding's copy of SRFTKV_STATIC_SCRATCH_BYTES is the header's value."""
    text = open(HEADER).read()
    m = re.search(r"#define\s+SRFTKV_STATIC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m, "SRFTKV_STATIC_SCRATCH_BYTES not found in the header"
    assert K.STATIC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))
