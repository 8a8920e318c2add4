"""GPU parity of the lighter scale planes (fp16 and e8m0 scales, groups of 16
and 32) against the fp64 oracle, on both codec paths and in decode
attention.

The stored scale is a rounding of A/Q computed by each side from its own z
(fp32 on the GPU, fp64 in the oracle), so where A/Q lies within 1e-5 of a
rounding boundary of the format (an fp16 midpoint, or a power of two for
e8m0) the two may store neighbouring values.  Everywhere else the stored
scales are bit-exact; the codes are checked against the pre-round values
z / scale of the scale the GPU stored, with the usual 1e-4 band."""

import numpy as np
import pytest
import torch

from oracle import srft_oracle as O
from int8_kv_cache_srft_gb300 import inputs as I
from tests.parity import ATTN_ATOL, assert_codes, assert_dequant_within_step

pytestmark = pytest.mark.gpu

K = None


@pytest.fixture(scope="module", autouse=True)
def _lib():
    global K
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import int8_kv_cache_srft_gb300 as mod

    mod.library()
    K = mod
    yield
    assert K.srftkv_device_fault() == 0


def _np(t):
    return t.detach().cpu().numpy()


def tm(t):
    return t.permute(0, 2, 1, 3)


def raw_np(scales: torch.Tensor, fmt: str) -> np.ndarray:
    t = _np(tm(scales))
    return t.view(np.uint16) if fmt == "fp16" else t


def near_boundary(a_over_q: np.ndarray, fmt: str, tol=1e-5) -> np.ndarray:
    """A/Q within tol (relative) of a rounding boundary of the format."""
    a = np.asarray(a_over_q, dtype=np.float64)
    if fmt == "e8m0":
        p = np.ldexp(1.0, np.round(np.log2(np.where(a > 0, a, 1.0))).astype(np.int64))
        return (a > 0) & (np.abs(a - p) <= tol * a)
    h16 = np.clip(a, 0, O.FP16_MAX).astype(np.float16)
    h = h16.astype(np.float64)
    below = np.where(h <= a, h, np.nextafter(h16, np.float16(-np.inf)).astype(np.float64))
    above = np.where(h >= a, h, np.nextafter(h16, np.float16(np.inf)).astype(np.float64))
    return (a > 0) & (np.abs(a - (below + above) / 2) <= tol * a)


def check_side(side, x, lam, bits, group, seed, fmt, transform="srft"):
    n, T, H, d = x.shape
    lam_b = None if lam is None else _np(lam)[:, None, :, :]
    enc = O.srft_kv_quantize(_np(x).astype(np.float64), lam_b, bits, group, seed, transform=transform,
                             scale_format=fmt)
    raw = raw_np(side.scales, fmt)[:, :T]
    want = np.asarray(enc["scales_raw"])
    diff = raw != want
    assert not (diff & ~near_boundary(enc["a_over_q"], fmt)).any(), "stored scales differ away from a boundary"
    if diff.any():  # the neighbouring value only
        assert np.abs(raw.astype(np.int64) - want.astype(np.int64))[diff].max() <= 1
    sc_gpu = np.repeat(O.decode_scales(raw, fmt), group, axis=-1)
    r_gpu = np.where(sc_gpu > 0, enc["z"] / np.where(sc_gpu > 0, sc_gpu, 1.0), 0.0)
    assert_codes(_np(tm(side.codes))[:, :T], r_gpu, bits)
    return enc, lam_b, raw


def encode(w, bits, group, fmt, seed, transform="srft"):
    xk = I.kv_side(w, "k")
    lk = I.lam_table(w, "k")
    n, T, H, d = xk.shape
    s = K.alloc_side(n, T, H, d, bits, group, transform=transform, scale_format=fmt)
    s.x = xk.cuda()
    s.lam = None if lk is None else lk.cuda()
    K.srft_kv_quantize(s, None, n, T, H, d, group, T, 0, seed)
    torch.cuda.synchronize()
    return s, xk, lk


CODEC = [(d, bits, group, fmt, path) for d in (16, 32, 64, 128, 256) for bits in (4, 8)
         for group in sorted({16, min(32, d)}) for fmt in ("fp16", "e8m0") for path in ("fft", "tc")
         if path == "fft" or d == 128]


@pytest.mark.parametrize("d,bits,group,fmt,path", CODEC)
def test_codec_scale_formats(monkeypatch, d, bits, group, fmt, path):
    monkeypatch.setenv("SRFTKV_QUANT_PATH", path)
    w = I.Workload("sf", n_outer=2, tokens=300, kv_heads=3, d=d, lam=(bits == 4), data_seed=3 * d + bits + group,
                   outlier_kind="scale", outlier_channels=2, outlier_factor=30.0)
    s, x, lam = encode(w, bits, group, fmt, 19)
    enc, lam_b, raw = check_side(s, x, lam, bits, group, 19, fmt)
    n, T, H, _ = x.shape
    out = torch.empty_like(s.x)
    K.srft_kv_dequantize(K.Side(s.codes, s.scales, bits, x=out, lam=s.lam, scale_format=fmt), None, n, T, H, d, group,
                         T, 0, 19)
    torch.cuda.synchronize()
    # the GPU decode of the GPU's codes and scales against the oracle decode of the same
    mine = O.srft_kv_dequantize(_np(tm(s.codes)), O.decode_scales(raw, fmt), lam_b, bits, group, 19)
    assert np.abs(_np(out) - mine).max() <= np.abs(mine).max() * 2.0**-10 + 1e-5
    lam_full = None if lam_b is None else np.broadcast_to(lam_b, x.shape)
    ref_hat = O.srft_kv_dequantize(enc["codes"], enc["scales"], lam_b, bits, group, 19)
    assert_dequant_within_step(_np(out), ref_hat, np.maximum(enc["scales"], O.decode_scales(raw, fmt)), lam_full,
                               group)


def test_e8m0_zero_groups_store_byte_zero():
    x = torch.zeros((1, 64, 2, 128), dtype=torch.float16)
    s = K.alloc_side(1, 64, 2, 128, 4, 16, scale_format="e8m0")
    s.x = x.cuda()
    K.srft_kv_quantize(s, None, 1, 64, 2, 128, 16, 64, 0, 3)
    torch.cuda.synchronize()
    assert not _np(s.scales).any() and not _np(s.codes).any()


@pytest.mark.parametrize("fmt_k,fmt_v", (("fp16", "fp16"), ("e8m0", "e8m0"), ("fp32", "e8m0"), ("fp16", "fp32")))
@pytest.mark.parametrize("d,group", ((64, 16), (128, 16), (128, 32), (256, 16)))
def test_attention_scale_formats(fmt_k, fmt_v, d, group):
    B, Hkv, rep, t_cap, seed = 2, 2, 4, 320, 31
    w = I.Workload("attn", n_outer=B, tokens=t_cap, kv_heads=Hkv, d=d, lam=True, data_seed=d + group,
                   outlier_kind="scale", outlier_channels=2, outlier_factor=8.0)
    sides = []
    for name, fmt in (("k", fmt_k), ("v", fmt_v)):
        x, lam = I.kv_side(w, name), I.lam_table(w, name)
        s = K.alloc_side(B, t_cap, Hkv, d, 4, group, scale_format=fmt)
        s.x, s.lam = x.cuda(), lam.cuda()
        K.srft_kv_quantize(s, None, B, t_cap, Hkv, d, group, t_cap, 0, seed)
        sides.append(s)
    torch.cuda.synchronize()
    q = I.query(I.Workload("q", n_outer=B, tokens=1, kv_heads=Hkv, d=d, q_heads=Hkv * rep, data_seed=d), device="cuda")
    seq = torch.tensor([320, 97], dtype=torch.int32, device="cuda")
    out = torch.empty((B, Hkv * rep, d), dtype=torch.float32, device="cuda")
    ws = torch.empty(K.q4kv_decode_attention_workspace_size(B, Hkv * rep, Hkv, d, t_cap, 0), dtype=torch.uint8,
                     device="cuda")
    K.q4kv_decode_attention(q, out, sides[0], sides[1], B, Hkv * rep, Hkv, d, group, t_cap, seq, 0.0, seed, 0, ws)
    torch.cuda.synchronize()

    def oside(s, fmt):
        return {"bits": 4, "codes": _np(tm(s.codes)), "scales": O.decode_scales(raw_np(s.scales, fmt), fmt),
                "lam": _np(s.lam).astype(np.float64), "group": group}

    ref = O.packed_decode_attention(_np(q).astype(np.float64), oside(sides[0], fmt_k), oside(sides[1], fmt_v), seed,
                                    _np(seq))
    assert np.abs(_np(out) - ref).max() <= ATTN_ATOL
