"""GPU parity of the tensor-core quantize at the wide head dimensions d = 192
(one CTA holds all of R_s) and d = 256 (CTA pairs split the output
coordinates) against the fp64 oracle, through the C ABI.

The tensor-core path is forced on (SRFTKV_QUANT_PATH=tc) for small ragged
calls: tiles of 128 tokens with a ragged last one, written at an offset of
a larger cache, rows outside the window checked untouched; every K/V width
pair, groups of 16 and 32, with and without lambda, fp32 / fp16 / e8m0 scale
planes, the Hadamard variant at d = 256, and a call of several hundred tiles
(several rounds of the persistent schedule).  The codes then go back through
the dequantize and are compared with the oracle's decode of the same codes.
"""

import numpy as np
import pytest
import torch

from oracle import srft_oracle as O
from int8_kv_cache_srft_gb300 import inputs as I
from tests.parity import assert_codes, assert_scales
from tests.test_gpu_scale_formats import near_boundary

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
    """Token-major view [outer][token][head][...] of a head-major plane [outer][head][token][...]."""
    return t.permute(0, 2, 1, 3)


def _quantize(xk, xv, lk, lv, bk, bv, group, seed, t_cap, t_offset, transform="srft", fmt="fp32"):
    n, T, H, d = xk.shape
    sides = []
    for x, lam, bits in ((xk, lk, bk), (xv, lv, bv)):
        s = K.alloc_side(n, t_cap, H, d, bits, group, transform=transform, scale_format=fmt)
        s.codes.fill_(0xAB)
        if fmt == "fp32":
            s.scales.fill_(-1.0)
        s.x = x.cuda()
        s.lam = None if lam is None else lam.cuda()
        sides.append(s)
    K.srft_kv_quantize(sides[0], sides[1], n, T, H, d, group, t_cap, t_offset, seed)
    torch.cuda.synchronize()
    return sides


def _check(side, x, lam, bits, group, seed, t_offset, transform="srft", fmt="fp32"):
    n, T, H, d = x.shape
    lam_b = None if lam is None else _np(lam)[:, None, :, :]
    enc = O.srft_kv_quantize(_np(x).astype(np.float64), lam_b, bits, group, seed, transform=transform,
                             scale_format=fmt)
    codes = _np(tm(side.codes))
    if fmt == "fp32":
        assert_scales(_np(tm(side.scales))[:, t_offset:t_offset + T], enc["scales"])
        assert_codes(codes[:, t_offset:t_offset + T], enc["r"], bits)
        scales = _np(tm(side.scales))[:, t_offset:t_offset + T].astype(np.float64)
    else:
        raw = _np(tm(side.scales))[:, t_offset:t_offset + T]
        raw = raw.view(np.uint16) if fmt == "fp16" else raw
        want = np.asarray(enc["scales_raw"])
        # stored scales may be neighbouring values only within 1e-5 of a rounding boundary of the format
        diff = raw != want
        assert not (diff & ~near_boundary(enc["a_over_q"], fmt)).any(), "stored scales differ away from a boundary"
        assert (np.abs(raw.astype(np.int64) - want.astype(np.int64)) <= 1).all()
        scales = O.decode_scales(raw, fmt)
        sc = np.repeat(scales, group, axis=-1)
        r = np.where(sc > 0, enc["z"] / np.where(sc > 0, sc, 1.0), 0.0)
        assert_codes(codes[:, t_offset:t_offset + T], r, bits)
    assert (codes[:, :t_offset] == 0xAB).all() and (codes[:, t_offset + T:] == 0xAB).all(), \
        "rows outside the window were written"
    return codes[:, t_offset:t_offset + T], scales, lam_b


def _roundtrip(side, codes, scales, lam_b, bits, group, seed, n, T, H, d, t_cap, t_offset, transform="srft",
               fmt="fp32"):
    out = torch.empty((n, T, H, d), dtype=torch.float16, device="cuda")
    K.srft_kv_dequantize(K.Side(side.codes, side.scales, bits, x=out, lam=side.lam, transform=transform,
                                scale_format=fmt), None, n, T, H, d, group, t_cap, t_offset, seed)
    torch.cuda.synchronize()
    mine = O.srft_kv_dequantize(codes, scales, lam_b, bits, group, seed, transform=transform)
    assert np.abs(_np(out) - mine).max() <= np.abs(mine).max() * 2.0**-10 + 1e-5


CASES = [(d, bk, bv, group, lam) for d in (192, 256) for bk, bv in ((4, 4), (8, 8), (8, 4), (4, 8))
         for group in (16, 32) for lam in (False, True)]


@pytest.mark.parametrize("d,bk,bv,group,lam", CASES)
def test_wide_tensor_core_quantize(monkeypatch, d, bk, bv, group, lam):
    """2 outer x 300 tokens x 3 heads (3 tiles of 128 a head, the last ragged) at t_offset 3 of t_cap 310."""
    monkeypatch.setenv("SRFTKV_QUANT_PATH", "tc")
    w = I.Workload("wide", n_outer=2, tokens=300, kv_heads=3, d=d, lam=lam, data_seed=d + bk * 10 + bv + group,
                   outlier_kind="scale", outlier_channels=4, outlier_factor=50.0)
    xk, xv = I.kv_side(w, "k"), I.kv_side(w, "v")
    lk, lv = I.lam_table(w, "k"), I.lam_table(w, "v")
    seed = 31
    sk, sv = _quantize(xk, xv, lk, lv, bk, bv, group, seed, 310, 3)
    for side, x, lam_t, b in ((sk, xk, lk, bk), (sv, xv, lv, bv)):
        codes, scales, lam_b = _check(side, x, lam_t, b, group, seed, 3)
        monkeypatch.setenv("SRFTKV_QUANT_PATH", "fft")  # the dequantize of these sizes: the register path
        _roundtrip(side, codes, scales, lam_b, b, group, seed, 2, 300, 3, d, 310, 3)
        monkeypatch.setenv("SRFTKV_QUANT_PATH", "tc")


@pytest.mark.parametrize("d,fmt", [(192, "fp16"), (192, "e8m0"), (256, "fp16"), (256, "e8m0")])
def test_wide_tensor_core_scale_formats(monkeypatch, d, fmt):
    monkeypatch.setenv("SRFTKV_QUANT_PATH", "tc")
    w = I.Workload("widef", n_outer=2, tokens=300, kv_heads=3, d=d, lam=True, data_seed=d + len(fmt),
                   outlier_kind="scale", outlier_channels=4, outlier_factor=50.0)
    xk, xv = I.kv_side(w, "k"), I.kv_side(w, "v")
    lk, lv = I.lam_table(w, "k"), I.lam_table(w, "v")
    for group in (16, 32):
        sk, sv = _quantize(xk, xv, lk, lv, 4, 8, group, 33, 310, 3, fmt=fmt)
        for side, x, lam_t, b in ((sk, xk, lk, 4), (sv, xv, lv, 8)):
            codes, scales, lam_b = _check(side, x, lam_t, b, group, 33, 3, fmt=fmt)
            monkeypatch.setenv("SRFTKV_QUANT_PATH", "fft")
            _roundtrip(side, codes, scales, lam_b, b, group, 33, 2, 300, 3, d, 310, 3, fmt=fmt)
            monkeypatch.setenv("SRFTKV_QUANT_PATH", "tc")


@pytest.mark.parametrize("bk,bv", ((4, 4), (8, 4)))
def test_wide_tensor_core_srht_d256(monkeypatch, bk, bv):
    monkeypatch.setenv("SRFTKV_QUANT_PATH", "tc")
    w = I.Workload("wideh", n_outer=2, tokens=300, kv_heads=3, d=256, lam=True, data_seed=77 + bk,
                   outlier_kind="scale", outlier_channels=4, outlier_factor=50.0)
    xk, xv = I.kv_side(w, "k"), I.kv_side(w, "v")
    lk, lv = I.lam_table(w, "k"), I.lam_table(w, "v")
    sk, sv = _quantize(xk, xv, lk, lv, bk, bv, 16, 35, 310, 3, transform="srht")
    for side, x, lam_t, b in ((sk, xk, lk, bk), (sv, xv, lv, bv)):
        codes, scales, lam_b = _check(side, x, lam_t, b, 16, 35, 3, transform="srht")
        monkeypatch.setenv("SRFTKV_QUANT_PATH", "fft")
        _roundtrip(side, codes, scales, lam_b, b, 16, 35, 2, 300, 3, 256, 310, 3, transform="srht")
        monkeypatch.setenv("SRFTKV_QUANT_PATH", "tc")


@pytest.mark.parametrize("d", (192, 256))
def test_wide_tensor_core_many_tiles(d):
    """4 outer x 5000 tokens x 4 heads (40 tiles a head, 1280 tiles over both sides: several rounds of the
    persistent schedule, above the automatic path's threshold): sampled rows against the oracle, plus every
    row by the reconstruction bound through the dequantize."""
    n, T, H, seed = 4, 5000, 4, 37
    w = I.Workload("widem", n_outer=n, tokens=T, kv_heads=H, d=d, data_seed=d + 1)
    xk, xv = I.kv_side(w, "k", device="cuda"), I.kv_side(w, "v", device="cuda")
    sk, sv = K.alloc_side(n, T, H, d, 4, 16), K.alloc_side(n, T, H, d, 4, 16)
    sk.x, sv.x = xk, xv
    K.srft_kv_quantize(sk, sv, n, T, H, d, 16, T, 0, seed)
    torch.cuda.synchronize()
    gen = np.random.default_rng(d)
    for side, x in ((sk, xk), (sv, xv)):
        o, t, h = gen.integers(0, n, 2000), gen.integers(0, T, 2000), gen.integers(0, H, 2000)
        oi, ti, hi = (torch.from_numpy(a).cuda() for a in (o, t, h))
        enc = O.srft_kv_quantize(_np(x[oi, ti, hi]).astype(np.float64)[:, None, :], None, 4, 16, seed)
        assert_scales(_np(side.scales[oi, hi, ti])[:, None, :], enc["scales"])
        assert_codes(_np(side.codes[oi, hi, ti])[:, None, :], enc["r"], 4)
        assert bool((side.scales > 0).all()), "unwritten scale rows"


DQ_CASES = [(d, bk, bv, group, fmt) for d in (192, 256) for bk, bv in ((4, 4), (8, 8), (8, 4), (4, 8))
            for group in (16, 32) for fmt in ("fp32", "fp16", "e8m0")]


@pytest.mark.parametrize("d,bk,bv,group,fmt", DQ_CASES)
def test_wide_tensor_core_dequantize(monkeypatch, d, bk, bv, group, fmt):
    """The tensor-core dequantize at d = 192 / 256 (forced on): codes written at t_offset 16 of t_cap 416 (so
    fp16 / e8m0 scale rows start on whole 16-byte rows), 2 outer x 300 tokens x 3 heads (ragged last tile),
    against the oracle's decode of the GPU's codes and within one quantisation step of the oracle's own."""
    w = I.Workload("widedq", n_outer=2, tokens=300, kv_heads=3, d=d, data_seed=d + 3 * bk + bv + group + len(fmt),
                   outlier_kind="scale", outlier_channels=4, outlier_factor=50.0)
    xk, xv = I.kv_side(w, "k"), I.kv_side(w, "v")
    monkeypatch.setenv("SRFTKV_QUANT_PATH", "tc")
    sk, sv = _quantize(xk, xv, None, None, bk, bv, group, 39, 416, 16, fmt=fmt)
    ok_, ov_ = torch.empty((2, 300, 3, d), dtype=torch.float16, device="cuda"), torch.empty(
        (2, 300, 3, d), dtype=torch.float16, device="cuda")
    ok_.fill_(float("nan"))
    ov_.fill_(float("nan"))
    K.srft_kv_dequantize(K.Side(sk.codes, sk.scales, bk, x=ok_, scale_format=fmt),
                         K.Side(sv.codes, sv.scales, bv, x=ov_, scale_format=fmt), 2, 300, 3, d, group, 416, 16, 39)
    torch.cuda.synchronize()
    for side, out, x, b in ((sk, ok_, xk, bk), (sv, ov_, xv, bv)):
        codes, scales, _ = _check(side, x, None, b, group, 39, 16, fmt=fmt)
        got = _np(out).astype(np.float64)
        assert np.isfinite(got).all()
        mine = O.srft_kv_dequantize(codes, scales, None, b, group, 39)
        assert np.abs(got - mine).max() <= np.abs(mine).max() * 2.0**-10 + 1e-5
